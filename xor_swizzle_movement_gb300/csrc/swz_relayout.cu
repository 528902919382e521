// swz_relayout.cu -- batched tile relayout between logical row-major order and
// Swizzle<B,M,S> physical order (sm_103a).
//
// Both directions are written as a gather over DESTINATION elements, so every
// thread stores to consecutive 16-byte vectors:
//   inverse  dst[i] = src[sw(i)]            -> source of y is sw(y)
//   forward  dst[sw(i)] = src[i]            -> source of y is sw^-1(y)
// (sw^-1 == sw when S >= B; otherwise the unitriangular inverse, see sw_inv.)
//
// Why a 16-byte vector always maps to ONE source vector (S > 0, or S < 0 with
// M >= log2 V): bit p of sw(x) (and of sw^-1(x)) depends only on bits p and
// above of x, because the field that is read (starting at M + S, S >= 1) sits
// above the field that is written.
// So the bits of the source offset at and above log2(16 / esize) depend only
// on the same bits of the destination offset: all lanes of a destination
// vector come from one source vector, permuted inside it.  The kernel is one
// 16-byte load, an in-register lane permutation, one 16-byte store.  A warp's
// 32 source vectors are a permutation of one aligned 512-byte block (the bits
// above the warp's span are again only read), so loads stay coalesced.
//
// The in-register lane permutation has three forms, chosen on the host:
//   kLanesFixed   M >= log2 V: groups of 2^M elements cover whole vectors,
//                 the lanes are not moved at all;
//   kLanesXor     M + S >= log2 V: the XOR constant is the same for every lane
//                 of the vector, the permutation is lane -> lane ^ L;
//   kLanesGeneral otherwise: the swizzle and its inverse are linear maps over
//                 GF(2) on the offset bits, and a vector's offset y (aligned)
//                 and its lane index l share no bit, so the source of lane l is
//                 g(y) ^ g(l): a per-vector constant k = g(y) mod V XOR-ed with
//                 a lane map L(l) = g(l) that is the same for every vector.
//                 The kernel first XORs the lanes by k (as kLanesXor), then
//                 applies the fixed permutation L as a byte permutation of the
//                 16-byte vector: three prmt per output word with selectors the
//                 host computes once per launch.
//
// Other requests (relayout_launch picks the path):
//   tiles of 1-8 bytes that divide 16: every vector holds whole tiles, so the
//     same kernel runs with the identity at vector level and one fixed lane map;
//   tiles that are not whole 16-byte vectors but hold whole swizzle periods,
//     on a buffer of whole vectors and aligned pointers: one tile (the swizzle
//     is the same on whole-buffer offsets);
//   other tiles that are not whole 16-byte vectors, aligned pointers: the
//     staged kernel (blocks of whole tiles in shared memory, 16-byte output
//     vectors gathered through a per-CTA table of their sources);
//   negative shifts whose read field lies below the lane bits (they split
//     vectors): a fixed lane map, warp shuffles within blocks of 32 vectors
//     (relayout_warp_coset_kernel), cosets of whole vectors in registers
//     (relayout_coset_kernel, relayout_coset_map_kernel), the staged kernel
//     over closure blocks, or element by element;
//   pointers aligned to the element size but not to 16 bytes: the vector
//     kernel on shifted pairs of aligned chunks (relayout_vec_mis_kernel) for
//     tiles of whole vectors, else the staged kernel staged at the pointers'
//     offsets, else element by element.
#include "swz_common.cuh"

#include <algorithm>
#include <cstring>

namespace swz {
namespace {

enum LaneMode { kLanesFixed = 0, kLanesXor = 1, kLanesGeneral = 2 };

struct RelayoutArgs {
    uint4 *dst;
    const uint4 *src;
    int64_t nvec;       // 16-byte vectors in the whole buffer
    int64_t tile_vecs;  // 16-byte vectors per tile
    int B, M, S;
    int steps;          // 1: source = sw(y); >1: source = sw^-1(y) by `steps` iterations
    int per_thread;     // vectors per thread, 1..kMaxPerThread
    uint32_t perm_sel[12];  // kLanesGeneral: prmt selectors of the fixed lane map L, 3 per word
};

constexpr int kMaxPerThread = 4;


// LINK: the variant for host-resident buffers, whose grid is sized for the
// host link: the grid walks the buffer in strides of itself, and loads carry
// no L2 eviction hint (with the evict-first hint a host-reading launch beside
// a host-writing one moved 12% less over the link).  Otherwise one CTA covers
// one stretch of blockDim.x * per_thread vectors, loads marked evict-first.
template <int E, int MODE, bool LOCAL, bool LINK>
__global__ void __launch_bounds__(256) relayout_vec_kernel(const RelayoutArgs a) {
    constexpr int LV = VecTraits<E>::LV;
    constexpr uint64_t VM = (1u << LV) - 1u;
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const int64_t step = LINK ? static_cast<int64_t>(gridDim.x) * blockDim.x * a.per_thread : a.nvec;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * a.per_thread + threadIdx.x; base < a.nvec;
         base += step) {
        uint4 r[kMaxPerThread];
        uint32_t lx[kMaxPerThread];
        const uint64_t policy = l2_evict_first_policy();
        // all loads first, so that each thread keeps up to kMaxPerThread 16-byte loads in flight
#pragma unroll
        for (int k = 0; k < kMaxPerThread; ++k) {
            const int64_t u = base + static_cast<int64_t>(k) * blockDim.x;
            if (k < a.per_thread && u < a.nvec) {
                int64_t local = u, tile0 = 0;
                if constexpr (LOCAL) {
                    local = u % a.tile_vecs;
                    tile0 = u - local;
                }
                const uint64_t y = static_cast<uint64_t>(local) << LV;
                const uint64_t x = sw_inv(y, a.B, a.M, a.S, a.steps);
                const uint4 *p = a.src + tile0 + static_cast<int64_t>(x >> LV);
                r[k] = LINK ? ld_stream16(p) : ld_stream16_hint(p, policy);
                lx[k] = static_cast<uint32_t>(x & VM);
            }
        }
#pragma unroll
        for (int k = 0; k < kMaxPerThread; ++k) {
            const int64_t u = base + static_cast<int64_t>(k) * blockDim.x;
            if (k < a.per_thread && u < a.nvec) {
                uint4 out;
                if constexpr (MODE == kLanesFixed) out = r[k];
                else if constexpr (MODE == kLanesXor) out = lanes_xor<E>(r[k], lx[k]);
                else out = bytes_permute(lanes_xor<E>(r[k], lx[k]), a.perm_sel);
                st_stream16(a.dst + u, out);
            }
        }
    }
}

// Bytes n .. n + 15 of the 32 bytes lo:hi (0 <= n < 16, n uniform over the
// launch): word selects and funnel shifts, no local memory.
__device__ __forceinline__ uint4 bytes_from_pair(uint4 lo, uint4 hi, int n) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const int q = n >> 2, r = (n & 3) * 8;
    uint32_t sel[5];
#pragma unroll
    for (int j = 0; j < 5; ++j) {
        const uint32_t a0 = w[j], a1 = w[j + 1], a2 = w[j + 2], a3 = w[j + 3 < 8 ? j + 3 : 7];
        sel[j] = q == 0 ? a0 : q == 1 ? a1 : q == 2 ? a2 : a3;
    }
    return make_uint4(__funnelshift_r(sel[0], sel[1], r), __funnelshift_r(sel[1], sel[2], r),
                      __funnelshift_r(sel[2], sel[3], r), __funnelshift_r(sel[3], sel[4], r));
}

// 16-byte load through L1 (allocating): for the pairs of aligned chunks that
// cover misaligned source vectors, where a lane's second chunk is mostly
// another lane's first.
__device__ __forceinline__ uint4 ld_l1_16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint8_t byte_of(const uint4 &v, int i) {
    const uint32_t w = i < 4 ? v.x : i < 8 ? v.y : i < 12 ? v.z : v.w;
    return static_cast<uint8_t>(w >> ((i & 3) * 8));
}

// The vector kernel for buffers whose pointers are aligned to the element
// size but not to 16 bytes (a_src, a_dst: their offsets within a 16-byte
// chunk, uniform).  Source: the two aligned chunks that cover a source vector,
// shifted by a_src bytes (the buffer's first and last vectors are read byte by
// byte, so no chunk outside the buffer is touched).  The chunks are loaded
// through L1: a lane's second chunk is mostly the first of the lane whose
// vector follows, so about half the pair's requests stop in L1 (with both
// loads bypassing L1, 64 x 64 16-bit tiles with the source 2 bytes off ran at
// 0.90 of the copy bandwidth against 0.96 now).
// Destination (DMIS, a_dst != 0): vector u straddles aligned chunks u and
// u + 1 (counted from dst - a_dst).  A warp takes groups of 32 consecutive
// vectors that overlap by one (group g starts at vector 31 g): lanes 0..30
// each store aligned chunk u + 1 whole, from their own vector's tail and the
// next lane's head (a shuffle), and lane 31 only lends its vector.  Every
// aligned chunk is then written once by one 16-byte store; only the buffer's
// first and last vectors write their outer part byte by byte.  (A mapping of
// 32 disjoint vectors per warp needs a 33rd vector for the last chunk, loaded
// by one lane on its own; with it, 64 MiB of 16-bit tiles ran at 4.4 TB/s
// against 6.8 now, destination + 2 bytes.)
// Without DMIS each lane stores its vector's aligned chunk directly.  Either
// way a warp walks per_thread consecutive groups.
template <int E, int MODE, bool LOCAL, bool DMIS>
__global__ void __launch_bounds__(256) relayout_vec_mis_kernel(const RelayoutArgs a, int a_src, int a_dst) {
    constexpr int LV = VecTraits<E>::LV;
    constexpr uint64_t VM = (1u << LV) - 1u;
    constexpr int kStep = DMIS ? 31 : 32;  // new vectors per warp group
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const uint8_t *srcb = reinterpret_cast<const uint8_t *>(a.src);
    uint8_t *dstb = reinterpret_cast<uint8_t *>(a.dst);
    const uint4 *sal = reinterpret_cast<const uint4 *>(srcb - a_src);
    uint4 *dal = reinterpret_cast<uint4 *>(dstb - a_dst);
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    // the source vector of destination vector u, its lanes not yet moved
    auto load_vec = [&](int64_t u, uint32_t &lxo) -> uint4 {
        int64_t local = u, tile0 = 0;
        if constexpr (LOCAL) {
            local = u % a.tile_vecs;
            tile0 = u - local;
        }
        const uint64_t y = static_cast<uint64_t>(local) << LV;
        const uint64_t x = sw_inv(y, a.B, a.M, a.S, a.steps);
        const int64_t sv = tile0 + static_cast<int64_t>(x >> LV);
        lxo = static_cast<uint32_t>(x & VM);
        if (a_src == 0) return ld_stream16(sal + sv);
        if (sv == 0 || sv == a.nvec - 1) {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            for (int i = 0; i < 16; ++i) w[i >> 2] |= static_cast<uint32_t>(srcb[16 * sv + i]) << ((i & 3) * 8);
            return make_uint4(w[0], w[1], w[2], w[3]);
        }
        return bytes_from_pair(ld_l1_16(sal + sv), ld_l1_16(sal + sv + 1), a_src);
    };
    uint4 r[kMaxPerThread];
    uint32_t lx[kMaxPerThread];
#pragma unroll
    for (int k = 0; k < kMaxPerThread; ++k) {
        const int64_t u = (gwarp * a.per_thread + k) * kStep + lane;
        if (k < a.per_thread && u < a.nvec) r[k] = load_vec(u, lx[k]);
    }
#pragma unroll
    for (int k = 0; k < kMaxPerThread; ++k) {
        if (k >= a.per_thread) break;  // uniform
        const int64_t u = (gwarp * a.per_thread + k) * kStep + lane;
        const bool act = u < a.nvec;
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (act) {
            if constexpr (MODE == kLanesFixed) out = r[k];
            else if constexpr (MODE == kLanesXor) out = lanes_xor<E>(r[k], lx[k]);
            else out = bytes_permute(lanes_xor<E>(r[k], lx[k]), a.perm_sel);
        }
        if constexpr (!DMIS) {
            if (act) st_stream16(dal + u, out);
        } else {
            uint4 nxt;
            nxt.x = __shfl_down_sync(kFullMask, out.x, 1);
            nxt.y = __shfl_down_sync(kFullMask, out.y, 1);
            nxt.z = __shfl_down_sync(kFullMask, out.z, 1);
            nxt.w = __shfl_down_sync(kFullMask, out.w, 1);
            if (!act || lane == 31) continue;  // lane 31's vector is the next group's first
            const int head = 16 - a_dst;       // bytes of vector u in aligned chunk u
            if (u == 0)
                for (int i = 0; i < head; ++i) dstb[i] = byte_of(out, i);
            if (u + 1 < a.nvec) st_stream16(dal + u + 1, bytes_from_pair(out, nxt, head));
            else
                for (int i = head; i < 16; ++i) dstb[16 * u + i] = byte_of(out, i);
        }
    }
}

// Negative shifts whose read field starts below a vector's lane bits (M <
// log2 V) but whose written field lies at or above them (M + |S| >= log2 V).
// The gather map G (sw^-1 forward, sw inverse) then never changes a lane bit,
// and on the bits of an offset it is linear over GF(2).  For destination
// vector d and lane l the source element is G(dV) ^ G(l): lane l of vector
// Gv(d) ^ Gv(l), Gv(.) the vector part.  Gv(l) only depends on the g read-
// field bits inside the lanes (g = min(M + B, log2 V) - M); their images w_i
// = Gv(2^(M+i)) span a g-dimensional space W.  The destination vectors whose
// sources lie in one coset s0 ^ W form one coset d0 ^ W' (W' = Gv^-1(W), basis
// w'_i = Gv^-1(w_i), s0 = Gv(d0)), so a thread owns such a pair: it loads the
// 2^g vectors V_k = s0 ^ w(k) once and stores the 2^g vectors D_j = d0 ^ w'(j),
// lane l of D_j being lane l of V_{j ^ phi(l)}, phi(l) = (l >> M) mod 2^g.
// Each source and each destination vector is touched once.  Lanes move in
// units of U = esize * 2^M bytes, so the kernel is instantiated on (U, g).
// Threads enumerate the cosets by their representative with zeros at the
// pivot bits of W' (reduced echelon form): consecutive threads take
// consecutive vectors below the lowest pivot.  Tiles hold whole closure
// blocks (2^(M + |S| + B) elements, checked by the caller), so global offsets
// equal tile-local ones.
struct CosetArgs {
    uint4 *dst;
    const uint4 *src;
    int64_t n_cosets;   // cosets (16-byte vectors / 2^g); with SB > 0, threads (vectors / 2^(g + SB))
    int B, M, S, steps, lv;
    int pivot[4];       // ascending bit positions left zero in a coset's representative
    int sbase;          // SB > 0: first of the g + SB bits a thread's cosets leave to its slots
    uint64_t w[4];      // source side: w_i (vector offsets)
    uint64_t wd[4];     // destination side: w'_i
};

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// 32-byte global store (two 16-byte vectors; the address is 32-byte aligned)
__device__ __forceinline__ void st_stream32(void *p, const uint4 &a, const uint4 &b) {
    asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
                 "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}

// Word q of D_j (j, q compile-time after unrolling): its bytes come from
// lanes of the same word in V_{j ^ phi}, one unit of U bytes at a time.
template <int U, int G>
__device__ __forceinline__ uint32_t coset_word(const uint4 (&v)[1 << G], int j, int q) {
    constexpr int m = (1 << G) - 1;
    if constexpr (U >= 4) {
        return word_of(v[j ^ (((4 * q) / U) & m)], q);
    } else if constexpr (U == 2) {
        return __byte_perm(word_of(v[j ^ ((2 * q) & m)], q), word_of(v[j ^ ((2 * q + 1) & m)], q), 0x7610);
    } else {
        const uint32_t ab = __byte_perm(word_of(v[j ^ ((4 * q) & m)], q), word_of(v[j ^ ((4 * q + 1) & m)], q), 0x3250);
        const uint32_t cd = __byte_perm(word_of(v[j ^ ((4 * q + 2) & m)], q), word_of(v[j ^ ((4 * q + 3) & m)], q), 0x7210);
        return __byte_perm(ab, cd, 0x7610);
    }
}

// SB > 0 (fields disjoint, |S| >= B, with r = B - g >= 2 read-field bits
// above the lanes): those bits sit at the bottom of the vector index and Gv
// copies them into the region bits just above the pivots, so a warp whose
// lanes take consecutive destination vectors reads 2^r regions, 16 bytes from
// each sector.  A thread then owns 2^SB cosets, d0 = base | (c << |S|) for the
// SB region bits c, base's low SB (read) bits being tau.  Load slot c fetches
// coset c ^ tau, whose sources are base's run of vectors in one region, so
// each load instruction reads whole sectors; SB stages of conditional swaps
// (by the bits of tau) then put coset c in slot c, and each store
// instruction writes whole sectors too.
// ST32 (SB = 0): W' is spanned by the lowest g vector bits with w'_i = e_i,
// so a coset's destination vectors are one aligned block of 2^g vectors,
// stored with 32-byte accesses (destination 32-byte aligned): a warp
// instruction then writes whole sectors, where 16-byte stores at a 2^g-vector
// stride wrote half of each.  (Such cosets whose sources stay in a block of 32
// vectors go to relayout_warp_coset_kernel instead.)
template <int U, int G, int SB, bool ST32>
__global__ void __launch_bounds__(256) relayout_coset_kernel(const CosetArgs a) {
    constexpr int NV = 1 << G;
    constexpr int NC = SB > 0 ? (1 << SB) : (G >= 3) ? 1 : (8 >> G);  // cosets per thread
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const uint64_t pol = l2_evict_first_policy();  // every source vector is read once
    uint4 v[NC][NV];
    uint64_t d0[NC];
    if constexpr (SB > 0) {
        const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        if (t >= a.n_cosets) return;  // (counts threads here: 2^SB cosets each)
        const int sb = a.sbase, s = -a.S;
        const uint64_t base = (static_cast<uint64_t>(t) & ((1ull << sb) - 1ull)) |
                              ((static_cast<uint64_t>(t) >> sb) << (s + SB));
        const uint32_t tau = static_cast<uint32_t>(base) & (NC - 1);
        // every load first, then every store (a store is a compiler barrier)
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            d0[c] = base | (static_cast<uint64_t>(c) << s);
            const uint64_t cl = base | (static_cast<uint64_t>(c ^ tau) << s);
            const uint64_t s0 = sw_inv(cl << a.lv, a.B, a.M, a.S, a.steps) >> a.lv;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                uint64_t x = s0;
#pragma unroll
                for (int i = 0; i < G; ++i)
                    if ((k >> i) & 1) x ^= a.w[i];
                v[c][k] = ld_stream16_hint(a.src + x, pol);
            }
        }
        // slot c <- slot c ^ tau
#pragma unroll
        for (int i = 0; i < SB; ++i) {
            const bool f = (tau >> i) & 1u;
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                if (c & (1 << i)) continue;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const uint4 x = v[c][k], y = v[c | (1 << i)][k];
                    v[c][k] = f ? y : x;
                    v[c | (1 << i)][k] = f ? x : y;
                }
            }
        }
    } else {
        const int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * NC + threadIdx.x;
        // every load first, then every store (a store is a compiler barrier)
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const int64_t t = base + static_cast<int64_t>(c) * blockDim.x;
            if (t < a.n_cosets) {
                uint64_t d = static_cast<uint64_t>(t);
#pragma unroll
                for (int i = 0; i < G; ++i) {
                    const int p = a.pivot[i];
                    d = ((d >> p) << (p + 1)) | (d & ((1ull << p) - 1ull));
                }
                d0[c] = d;
                const uint64_t s0 = sw_inv(d << a.lv, a.B, a.M, a.S, a.steps) >> a.lv;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    uint64_t x = s0;
#pragma unroll
                    for (int i = 0; i < G; ++i)
                        if ((k >> i) & 1) x ^= a.w[i];
                    v[c][k] = ld_stream16_hint(a.src + x, pol);
                }
            }
        }
    }
    const int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * (SB > 0 ? 1 : NC) + threadIdx.x;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        if (SB == 0 && base + static_cast<int64_t>(c) * blockDim.x >= a.n_cosets) continue;
        if constexpr (ST32) {
#pragma unroll
            for (int j = 0; j < NV; j += 2) {
                uint4 o0, o1;
                o0.x = coset_word<U, G>(v[c], j, 0);
                o0.y = coset_word<U, G>(v[c], j, 1);
                o0.z = coset_word<U, G>(v[c], j, 2);
                o0.w = coset_word<U, G>(v[c], j, 3);
                o1.x = coset_word<U, G>(v[c], j + 1, 0);
                o1.y = coset_word<U, G>(v[c], j + 1, 1);
                o1.z = coset_word<U, G>(v[c], j + 1, 2);
                o1.w = coset_word<U, G>(v[c], j + 1, 3);
                st_stream32(a.dst + d0[c] + j, o0, o1);
            }
        } else {
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                uint64_t d = d0[c];
#pragma unroll
                for (int i = 0; i < G; ++i)
                    if ((j >> i) & 1) d ^= a.wd[i];
                uint4 o;
                o.x = coset_word<U, G>(v[c], j, 0);
                o.y = coset_word<U, G>(v[c], j, 1);
                o.z = coset_word<U, G>(v[c], j, 2);
                o.w = coset_word<U, G>(v[c], j, 3);
                st_stream16(a.dst + d, o);
            }
        }
    }
}

// Negative shifts that split vectors, where the gather map G keeps every
// destination vector's sources inside its own aligned block of 32 vectors:
// Gv preserves the block index on every vector bit, and the offset
// off(t) = Gv(unit t's first lane) of every unit of U = esize * 2^M bytes is
// below 32.  The source of unit t of destination vector u is then unit t of
// vector Gv(u) ^ off(t) after the fixed lane permutation Lam (the lane part of
// G; the identity when the written field lies at or above the lanes).  A warp
// loads its 32 destination positions' own vectors (one coalesced 512-byte load,
// as the plain relayout), permutes each by Lam when needed, and builds every
// output word from shuffles across the warp: lane Gv(u) ^ off(t) mod 32.
// Every global access is a whole 512-byte warp access, where the register
// coset kernels read a coset at a 2^p0-vector stride.  Lanes past the buffer's
// end take part in the shuffles without touching memory; no lane inside the
// buffer reads theirs (a source lies in its destination's closure block).
struct WarpCosetArgs {
    uint4 *dst;
    const uint4 *src;
    int64_t nvec;
    int B, M, S, steps, lv;
    int per_thread;
    uint32_t off[16];       // per unit: the source's vector offset, XOR-ed onto Gv(u) (below 32)
    uint32_t perm_sel[12];  // MAP: byte-permutation selectors of Lam (3 per word)
};

// Word q of an output vector from the warp's vectors: NB = 1, the block is
// the warp's 32 vectors (one register, v0); NB = 2, a block of 64 vectors,
// the lane's vectors in its two halves in v0 and v1 (two shuffles, then a
// select by bit 5 of the source position).
template <int U, int NB>
__device__ __forceinline__ uint32_t warp_coset_word(const uint4 &v0, const uint4 &v1, int q, uint32_t gl,
                                                    const uint32_t *off) {
    const uint32_t w0 = word_of(v0, q);
    const uint32_t w1 = NB == 2 ? word_of(v1, q) : 0u;
    auto from = [&](int t) -> uint32_t {
        const uint32_t x = gl ^ off[t];
        const uint32_t a0 = __shfl_sync(kFullMask, w0, static_cast<int>(x & 31u));
        if constexpr (NB == 1) {
            return a0;
        } else {
            const uint32_t a1 = __shfl_sync(kFullMask, w1, static_cast<int>(x & 31u));
            return (x & 32u) ? a1 : a0;
        }
    };
    if constexpr (U >= 4) {
        return from((4 * q) / U);
    } else if constexpr (U == 2) {
        return __byte_perm(from(2 * q), from(2 * q + 1), 0x7610);
    } else {
        const uint32_t ab = __byte_perm(from(4 * q), from(4 * q + 1), 0x3250);
        const uint32_t cd = __byte_perm(from(4 * q + 2), from(4 * q + 3), 0x7210);
        return __byte_perm(ab, cd, 0x7610);
    }
}

template <int U, bool MAP, int NB>
__global__ void __launch_bounds__(256) relayout_warp_coset_kernel(const WarpCosetArgs a) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const uint64_t pol = l2_evict_first_policy();
    const uint32_t lane = threadIdx.x & 31u;
    // Gv(u) mod 32 NB: a negative shift writes each read bit higher up, so the
    // bits of u above the block never reach Gv(u)'s position in the block, and
    // u's position in the block is the lane (plus 32 in a block's second half):
    // one value per half, per thread
    uint32_t gl[NB];
#pragma unroll
    for (int h = 0; h < NB; ++h)
        gl[h] = static_cast<uint32_t>(sw_inv(static_cast<uint64_t>(h * 32 + lane) << a.lv, a.B, a.M, a.S, a.steps) >>
                                      a.lv) &
                (32u * NB - 1u);
    // vector k of the thread: NB = 1, a stride of the CTA; NB = 2, the halves of
    // the warp's k / 2-th block of 64 (every load instruction covers 32
    // consecutive vectors either way)
    auto vec_index = [&](int k) -> int64_t {
        if constexpr (NB == 1) {
            return static_cast<int64_t>(blockIdx.x) * blockDim.x * a.per_thread + threadIdx.x +
                   static_cast<int64_t>(k) * blockDim.x;
        } else {
            const int64_t warp = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
            return (warp * (a.per_thread >> 1) + (k >> 1)) * 64 + (k & 1) * 32 + lane;
        }
    };
    uint4 v[kMaxPerThread];
#pragma unroll
    for (int k = 0; k < kMaxPerThread; ++k) {
        const int64_t u = vec_index(k);
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        if (k < a.per_thread && u < a.nvec) v[k] = ld_stream16_hint(a.src + u, pol);
    }
#pragma unroll
    for (int k = 0; k < kMaxPerThread; ++k) {
        if (k >= a.per_thread) break;  // uniform: every lane of the warp shuffles
        if constexpr (MAP) v[k] = bytes_permute(v[k], a.perm_sel);
    }
#pragma unroll
    for (int k = 0; k < kMaxPerThread; ++k) {
        if (k >= a.per_thread) break;
        const int64_t u = vec_index(k);
        const uint4 &v0 = NB == 1 ? v[k] : v[k & ~1];
        const uint4 &v1 = NB == 1 ? v[k] : v[k | 1];
        const uint32_t g = gl[NB == 1 ? 0 : (k & 1)];
        uint4 o;
        o.x = warp_coset_word<U, NB>(v0, v1, 0, g, a.off);
        o.y = warp_coset_word<U, NB>(v0, v1, 1, g, a.off);
        o.z = warp_coset_word<U, NB>(v0, v1, 2, g, a.off);
        o.w = warp_coset_word<U, NB>(v0, v1, 3, g, a.off);
        if (u < a.nvec) st_stream16(a.dst + u, o);
    }
}

// Negative shifts whose written field starts inside the lanes (M + |S| <
// log2 V < M + |S| + B).  The lane bits of G(y) still depend only on the lane
// bits of y, so G(dV) has no lane part and lane l of destination vector d
// comes from lane Lam(l) of vector Gv(d) ^ Gv(l): Lam, the lane part of G on
// a lane index, is a fixed permutation, and Gv(l) lies in the span W of the
// vector images of the lane bits (dimension g).  With phi(l) the coordinates
// of Gv(l) in a basis of W, destination D_j of a coset is the blend
// OR_m (Lam(V_(j ^ m)) & mask_m), mask_m the bytes of the lanes with phi = m
// (host-computed).  Cosets are enumerated as in relayout_coset_kernel.
struct CosetMapArgs {
    CosetArgs c;
    uint32_t perm_sel[12];  // byte-permutation selectors of Lam (3 per word)
    uint32_t mask[8][4];    // byte masks of the lanes with phi == m (m < 2^g)
};

// ST32 as for relayout_coset_kernel: 32-byte stores of the aligned
// destination block (the host picks the basis w'_i = e_i when W' is spanned by
// the lowest g vector bits).
template <int G, bool ST32>
__global__ void __launch_bounds__(256) relayout_coset_map_kernel(const CosetMapArgs a) {
    constexpr int NV = 1 << G;
    constexpr int NC = (G >= 3) ? 1 : (8 >> G);  // cosets per thread: 8 vectors in flight
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const uint64_t pol = l2_evict_first_policy();  // every source vector is read once
    const CosetArgs &c = a.c;
    const int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * NC + threadIdx.x;
    uint4 v[NC][NV];
    uint64_t d0[NC];
    // every load first, then every store (a store is a compiler barrier)
#pragma unroll
    for (int q = 0; q < NC; ++q) {
        const int64_t t = base + static_cast<int64_t>(q) * blockDim.x;
        if (t < c.n_cosets) {
            uint64_t d = static_cast<uint64_t>(t);
#pragma unroll
            for (int i = 0; i < G; ++i) {
                const int p = c.pivot[i];
                d = ((d >> p) << (p + 1)) | (d & ((1ull << p) - 1ull));
            }
            d0[q] = d;
            const uint64_t s0 = sw_inv(d << c.lv, c.B, c.M, c.S, c.steps) >> c.lv;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                uint64_t x = s0;
#pragma unroll
                for (int i = 0; i < G; ++i)
                    if ((k >> i) & 1) x ^= c.w[i];
                v[q][k] = ld_stream16_hint(c.src + x, pol);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < NC; ++q) {
        if (base + static_cast<int64_t>(q) * blockDim.x >= c.n_cosets) continue;
        // (a written bit lies inside the lanes, so Lam is never the identity)
#pragma unroll
        for (int k = 0; k < NV; ++k) v[q][k] = bytes_permute(v[q][k], a.perm_sel);
        uint4 o[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            o[j] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int m = 0; m < NV; ++m) {
                const uint4 x = v[q][j ^ m];
                o[j].x |= x.x & a.mask[m][0];
                o[j].y |= x.y & a.mask[m][1];
                o[j].z |= x.z & a.mask[m][2];
                o[j].w |= x.w & a.mask[m][3];
            }
        }
        if constexpr (ST32) {
#pragma unroll
            for (int j = 0; j < NV; j += 2) st_stream32(c.dst + d0[q] + j, o[j], o[j + 1]);
        } else {
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                uint64_t d = d0[q];
#pragma unroll
                for (int i = 0; i < G; ++i)
                    if ((j >> i) & 1) d ^= c.wd[i];
                st_stream16(c.dst + d, o[j]);
            }
        }
    }
}

template <int E>
struct ElemType;
template <> struct ElemType<1> { using T = uint8_t; };
template <> struct ElemType<2> { using T = uint16_t; };
template <> struct ElemType<4> { using T = uint32_t; };
template <> struct ElemType<8> { using T = uint2; };
template <> struct ElemType<16> { using T = uint4; };

// Element by element; used when a tile is not a whole number of 16-byte
// vectors or a pointer is not 16-byte aligned.  Each thread keeps four
// independent elements in flight, and tile-local offsets (a 64-bit remainder)
// are taken only when the tile does not hold whole swizzle periods.
template <int E, bool LOCAL>
__global__ void __launch_bounds__(256)
    relayout_scalar_kernel(void *dst, const void *src, int64_t n_elems, int64_t tile_elems, int B,
                           int M, int S, int steps) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    using T = typename ElemType<E>::T;
    constexpr int U = 4;
    T *d = static_cast<T *>(dst);
    const T *s = static_cast<const T *>(src);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n_elems;
         i0 += U * stride) {
        T v[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t i = i0 + k * stride;
            if (i < n_elems) {
                int64_t local = i, tile0 = 0;
                if constexpr (LOCAL) {
                    local = i % tile_elems;
                    tile0 = i - local;
                }
                const uint64_t x = sw_inv(static_cast<uint64_t>(local), B, M, S, steps);
                v[k] = s[tile0 + static_cast<int64_t>(x)];
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t i = i0 + k * stride;
            if (i < n_elems) d[i] = v[k];
        }
    }
}

// link_grid: a buffer lives in host memory.  The host link, not the SMs,
// bounds such a copy (about 0.2 TB/s each way, reached with a few dozen
// CTAs), so the grid is capped at 4 CTAs per SM and strides over the buffer:
// a relayout writing host memory on one stream then runs beside one reading
// it on another, and both directions of the link carry data at once.  A grid
// of one CTA per stretch would fill every SM until its last wave and
// serialise the two.  Such launches also go without programmatic dependent
// launch: the next kernel's CTAs would otherwise sit resident, waiting, in
// the slots the other stream's kernel needs.
template <int E>
swz_status launch_vec(const RelayoutArgs &a, int mode, bool local, bool link_grid, cudaStream_t st) {
    const int threads = 256;
    const int64_t per_cta = static_cast<int64_t>(threads) * a.per_thread;
    int64_t grid = (a.nvec + per_cta - 1) / per_cta;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 4;
    if (link_grid && grid > cap) grid = cap;
    if (grid > 0x7fffffffLL) return SWZ_ERR_SHAPE;
    const dim3 g(static_cast<unsigned>(grid));
#define SWZ_LAUNCH(MODE, LOCAL, LINK) \
    launch_pdl_if(!LINK, relayout_vec_kernel<E, MODE, LOCAL, LINK>, g, dim3(threads), 0, st, a)
#define SWZ_LAUNCH_MODES(LOCAL, LINK)                                         \
    (mode == kLanesFixed ? SWZ_LAUNCH(kLanesFixed, LOCAL, LINK)               \
     : mode == kLanesXor ? SWZ_LAUNCH(kLanesXor, LOCAL, LINK)                 \
                         : SWZ_LAUNCH(kLanesGeneral, LOCAL, LINK))
    cudaError_t e;
    if (local) e = link_grid ? SWZ_LAUNCH_MODES(true, true) : SWZ_LAUNCH_MODES(true, false);
    else e = link_grid ? SWZ_LAUNCH_MODES(false, true) : SWZ_LAUNCH_MODES(false, false);
#undef SWZ_LAUNCH_MODES
#undef SWZ_LAUNCH
    return launched(e);
}

// Tiles of whole 16-byte vectors on pointers aligned to the element size but
// not to 16 bytes: relayout_vec_mis_kernel, one CTA per stretch of vectors.
template <int E>
swz_status launch_vec_mis(const RelayoutArgs &a, int mode, bool local, int a_src, int a_dst, cudaStream_t st) {
    const int threads = 256;
    // a warp covers per_thread groups of 32 vectors, 31 new ones per group when dst is misaligned
    const int64_t per_cta = static_cast<int64_t>(threads / 32) * a.per_thread * (a_dst ? 31 : 32);
    const int64_t grid = (a.nvec + per_cta - 1) / per_cta;
    if (grid > 0x7fffffffLL) return SWZ_ERR_SHAPE;
    const dim3 g(static_cast<unsigned>(grid));
#define SWZ_LAUNCH(MODE, LOCAL)                                                                        \
    (a_dst ? launch_pdl(relayout_vec_mis_kernel<E, MODE, LOCAL, true>, g, dim3(threads), 0, st, a, a_src, a_dst) \
           : launch_pdl(relayout_vec_mis_kernel<E, MODE, LOCAL, false>, g, dim3(threads), 0, st, a, a_src, a_dst))
    cudaError_t e;
    if (local) e = mode == kLanesFixed ? SWZ_LAUNCH(kLanesFixed, true)
                   : mode == kLanesXor ? SWZ_LAUNCH(kLanesXor, true) : SWZ_LAUNCH(kLanesGeneral, true);
    else e = mode == kLanesFixed ? SWZ_LAUNCH(kLanesFixed, false)
             : mode == kLanesXor ? SWZ_LAUNCH(kLanesXor, false) : SWZ_LAUNCH(kLanesGeneral, false);
#undef SWZ_LAUNCH
    return launched(e);
}

// Tiles whose byte size is not a multiple of 16, with 16-byte aligned
// pointers: a CTA stages a block of whole tiles (a multiple of
// lcm(tile bytes, 16), at most kStageBytes) in shared memory with 16-byte
// loads; each thread then gathers one 16-byte output vector element by
// element from the staged block and stores it with one 16-byte store.  The
// block starts on a tile boundary, so an element's tile-local offset is its
// block offset modulo the tile: a multiply-high by a precomputed reciprocal
// (exact while offset x tile < 2^32) for a vector's first element, then a
// running count.
constexpr int kStageBytes = 8192;

// sw_inv on offsets below 2^16 in 32-bit arithmetic; the launcher passes
// B = 0 when the read field starts at or above bit 16 (the swizzle is then the
// identity on every offset of a staged block).
__device__ __forceinline__ uint32_t sw_inv32(uint32_t y, int B, int M, int S, int steps) {
    const uint32_t mask = (1u << B) - 1u;
    const int r = sw_read_lo(M, S), w = sw_write_lo(M, S);
    uint32_t x = y;
    for (int i = 0; i < steps; ++i) x = y ^ (((x >> r) & mask) << w);
    return x;
}

// MIS: dst or src is not 16-byte aligned (both are aligned to the element
// size).  The block is staged at its source's offset within a 16-byte chunk
// (a_src) by 16-byte loads of the aligned chunks that cover it, gathered into
// a second shared buffer at the destination's offset (a_dst), and written out
// by 16-byte stores of every aligned destination chunk the block owns whole.
// The chunk shared with the neighbouring block at each end goes out byte by
// byte (only this block's bytes), and chunks that reach past either end of
// the buffer are read byte by byte too.
template <int E, bool MIS>
__global__ void __launch_bounds__(256)
    relayout_staged_kernel(uint8_t *dst, const uint8_t *src, int64_t bytes, int block_bytes, uint32_t te,
                           uint32_t te_recip, uint32_t pat, uint32_t pat_recip, int B, int M, int S,
                           int steps, int a_src, int a_dst) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    using T = typename ElemType<E>::T;
    constexpr int V = 16 / E;  // elements per output vector
    __shared__ __align__(16) uint8_t a_s[kStageBytes + (MIS ? 16 : 0)];
    __shared__ __align__(16) uint8_t b_s[MIS ? kStageBytes + 16 : 16];
    // Source of each element of an output vector, relative to the vector's
    // first element.  Blocks start on multiples of lcm(tile bytes, 16), so the
    // pattern repeats every `pat` vectors; it is computed once per CTA.
    __shared__ __align__(16) int16_t rel_s[kStageBytes / E];
    const int tid = threadIdx.x;
    if (!MIS) a_src = a_dst = 0;
    auto local_of = [&](uint32_t e) -> uint32_t { return te == 1 ? 0u : e - __umulhi(e, te_recip) * te; };
    for (uint32_t i = tid; i < pat * V; i += 256) {
        const uint32_t local = local_of(i);
        rel_s[i] = static_cast<int16_t>(static_cast<int>(i - local + sw_inv32(local, B, M, S, steps)) -
                                        static_cast<int>(i));
    }
    __syncthreads();
    const uint8_t *sa = a_s + a_src;  // element-space byte j of the block is sa[j]
    for (int64_t b0 = static_cast<int64_t>(blockIdx.x) * block_bytes; b0 < bytes;
         b0 += static_cast<int64_t>(gridDim.x) * block_bytes) {
        const int nb = static_cast<int>(bytes - b0 < block_bytes ? bytes - b0 : block_bytes);
        const int nv = nb / 16;
        if constexpr (MIS) {
            // chunk q of a_s holds the element-space bytes b0 - a_src + 16q .. + 15
            const int nq = (a_src + nb + 15) / 16;
            for (int q = tid; q < nq; q += 256) {
                const int64_t g0 = b0 - a_src + 16 * q;
                if (g0 >= 0 && g0 + 16 <= bytes) {
                    *reinterpret_cast<uint4 *>(a_s + 16 * q) = ld_stream16(src + g0);
                } else {
                    for (int t = 0; t < 16; ++t)
                        if (g0 + t >= 0 && g0 + t < bytes) a_s[16 * q + t] = src[g0 + t];
                }
            }
        } else {
            for (int v = tid; v < nv; v += 256)
                *reinterpret_cast<uint4 *>(a_s + 16 * v) = ld_stream16(src + b0 + 16 * v);
            for (int t = 16 * nv + tid; t < nb; t += 256) a_s[t] = src[b0 + t];
        }
        __syncthreads();
        const uint32_t ne = static_cast<uint32_t>(nb / E);
        if constexpr (MIS) {
            // one unit per thread, consecutive units on consecutive lanes, so
            // that both the staged reads and the shared writes stay free of
            // bank conflicts (a vector per thread would put the lanes 16
            // bytes apart); the table repeats every pat * V units
            const uint32_t pv = pat * V;
            const uint32_t pv_recip = pv == 1 ? 0u : static_cast<uint32_t>((uint64_t(1) << 32) / pv + 1);
            for (uint32_t e = tid; e < static_cast<uint32_t>(nv) * V; e += 256) {
                const uint32_t i = pv == 1 ? 0u : e - __umulhi(e, pv_recip) * pv;
                *reinterpret_cast<T *>(b_s + a_dst + e * E) =
                    *reinterpret_cast<const T *>(sa + (static_cast<int>(e) + rel_s[i]) * E);
            }
        } else if constexpr (E == 1) {
            // 1-byte units: one 32-bit output word per thread, so that the
            // lanes of a warp read neighbouring staged bytes (a vector per
            // thread puts them 16 bytes apart: 4-way bank conflicts on every
            // byte load) and store 128 contiguous bytes per instruction.  (For
            // 2-byte units the same form measured 12% slower than a vector per
            // thread, which loads only 8 units per vector.)
            const uint32_t pw = pat * 4;  // words per period of the table
            const uint32_t pw_recip = pw == 1 ? 0u : static_cast<uint32_t>((uint64_t(1) << 32) / pw + 1);
            for (uint32_t w = tid; w < static_cast<uint32_t>(nv) * 4; w += 256) {
                const uint32_t i = pw == 1 ? 0u : w - __umulhi(w, pw_recip) * pw;
                const int e = static_cast<int>(w) * 4;
                const uint2 rr = *reinterpret_cast<const uint2 *>(rel_s + i * 4);  // the word's 4 table entries
                const int r0 = static_cast<int16_t>(rr.x & 0xffffu), r1 = static_cast<int16_t>(rr.x >> 16);
                const int r2 = static_cast<int16_t>(rr.y & 0xffffu), r3 = static_cast<int16_t>(rr.y >> 16);
                const uint32_t word = static_cast<uint32_t>(sa[e + r0]) | (static_cast<uint32_t>(sa[e + 1 + r1]) << 8) |
                                      (static_cast<uint32_t>(sa[e + 2 + r2]) << 16) |
                                      (static_cast<uint32_t>(sa[e + 3 + r3]) << 24);
                *reinterpret_cast<uint32_t *>(dst + b0 + 4 * w) = word;
            }
        } else {
            for (int v = tid; v < nv; v += 256) {
                const uint32_t e = static_cast<uint32_t>(v) * V;
                const uint32_t p = pat == 1 ? 0u : static_cast<uint32_t>(v) - __umulhi(static_cast<uint32_t>(v), pat_recip) * pat;
                int16_t rel[V];
                memcpy(rel, rel_s + p * V, sizeof rel);
                T lanes[V];
#pragma unroll
                for (int k = 0; k < V; ++k)
                    lanes[k] = *reinterpret_cast<const T *>(sa + (static_cast<int>(e + k) + rel[k]) * E);
                uint4 o;
                memcpy(&o, lanes, 16);
                st_stream16(dst + b0 + 16 * v, o);
            }
        }
        for (uint32_t e = static_cast<uint32_t>(nv) * V + tid; e < ne; e += 256) {
            const uint32_t local = local_of(e);
            const uint32_t x = sw_inv32(local, B, M, S, steps);
            const T val = *reinterpret_cast<const T *>(sa + (e - local + x) * E);
            if constexpr (MIS) *reinterpret_cast<T *>(b_s + a_dst + e * E) = val;
            else *reinterpret_cast<T *>(dst + b0 + e * E) = val;
        }
        if constexpr (MIS) {
            __syncthreads();
            // chunk q of b_s is the 16-byte aligned destination chunk at dst + b0 - a_dst + 16q;
            // this block owns its bytes a_dst .. a_dst + nb - 1
            const int nq = (a_dst + nb + 15) / 16;
            for (int q = tid; q < nq; q += 256) {
                const int t0 = 16 * q;
                if (t0 >= a_dst && t0 + 16 <= a_dst + nb) {
                    st_stream16(dst + b0 - a_dst + t0, *reinterpret_cast<const uint4 *>(b_s + t0));
                } else {
                    for (int t = t0; t < t0 + 16; ++t)
                        if (t >= a_dst && t < a_dst + nb) dst[b0 - a_dst + t] = b_s[t];
                }
            }
        }
        __syncthreads();  // the buffers are refilled for the next block
    }
}

template <int E, bool MIS>
swz_status launch_staged(void *dst, const void *src, int64_t bytes, int block_bytes, int64_t tile_elems, int B,
                         int M, int S, int steps, int a_src, int a_dst, cudaStream_t st) {
    if (tile_elems <= 0 || block_bytes <= 0) return SWZ_ERR_PARAM;
    int64_t grid = (bytes + block_bytes - 1) / block_bytes;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    if (grid > cap) grid = cap;
    const uint32_t te = static_cast<uint32_t>(tile_elems);
    const uint32_t recip = te == 1 ? 0u : static_cast<uint32_t>((uint64_t(1) << 32) / te + 1);
    // staged offsets are below kStageBytes <= 2^16: a read field at or above
    // bit 16 is all zero there, and the swizzle is the identity
    if (sw_read_lo(M, S) >= 16) { B = 0; M = 0; S = 1; steps = 1; }
    // the source pattern of output vectors repeats every lcm(tile bytes, 16) bytes
    int64_t g = te * E, h = 16;
    while (h) { const int64_t r = g % h; g = h; h = r; }
    const uint32_t pat = static_cast<uint32_t>(te * E / g);  // lcm / 16 vectors
    const uint32_t pat_recip = pat == 1 ? 0u : static_cast<uint32_t>((uint64_t(1) << 32) / pat + 1);
    return launched(launch_pdl(relayout_staged_kernel<E, MIS>, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st,
                               static_cast<uint8_t *>(dst), static_cast<const uint8_t *>(src), bytes, block_bytes,
                               te, recip, pat, pat_recip, B, M, S, steps, a_src, a_dst));
}

template <int E>
swz_status launch_scalar(void *dst, const void *src, int64_t n, int64_t tile, int B, int M, int S,
                         int steps, cudaStream_t st) {
    const int threads = 256;
    int64_t grid = (n + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 32;
    if (grid > cap) grid = cap;
    const int period = B + M + (S < 0 ? -S : S);  // the offset bits the swizzle touches
    const bool local = B > 0 && (period >= 62 || (tile & ((int64_t(1) << period) - 1)) != 0);
    const dim3 g(static_cast<unsigned>(grid));
    if (local)
        return launched(launch_pdl(relayout_scalar_kernel<E, true>, g, dim3(threads), 0, st, dst, src, n, tile, B,
                                   M, S, steps));
    return launched(launch_pdl(relayout_scalar_kernel<E, false>, g, dim3(threads), 0, st, dst, src, n, tile, B, M,
                               S, steps));
}

// Every 16-byte vector holds whole blocks of `te` elements that the swizzle
// maps onto themselves (te divides 16 / esize): each vector stays where it is
// and its lanes move by one fixed permutation.  The vector kernel runs with
// the identity at vector level (B = 0) and that permutation as its lane map.
swz_status launch_lane_map(void *dst, const void *src, int64_t n_elems, int esize, int te, int B, int M, int S,
                           int steps, bool link_grid, cudaStream_t st) {
    const int lanes = 16 / esize;
    int src_lane[16];
    for (int l = 0; l < lanes; ++l)
        src_lane[l] = (l - l % te) + static_cast<int>(sw_inv(static_cast<uint64_t>(l % te), B, M, S, steps));
    RelayoutArgs a;
    a.dst = static_cast<uint4 *>(dst);
    a.src = static_cast<const uint4 *>(src);
    a.nvec = n_elems * esize / 16;
    a.tile_vecs = 1;
    a.B = 0; a.M = 0; a.S = 1;
    a.steps = 1;
    const int64_t wave = static_cast<int64_t>(sm_count()) * 2048;
    a.per_thread = (a.nvec >= 4 * wave) ? 4 : (a.nvec >= 2 * wave) ? 2 : 1;
    lane_map_selectors(src_lane, esize, a.perm_sel);
    switch (esize) {
        case 1: return launch_vec<1>(a, kLanesGeneral, false, link_grid, st);
        case 2: return launch_vec<2>(a, kLanesGeneral, false, link_grid, st);
        case 4: return launch_vec<4>(a, kLanesGeneral, false, link_grid, st);
        default: return launch_vec<8>(a, kLanesGeneral, false, link_grid, st);
    }
}

// The staged kernel over blocks of whole `te`-element tiles (te * esize need
// not be a multiple of 16).  Pointers that are not 16-byte aligned take the
// kernel's MIS form.  Returns SWZ_ERR_UNSUPPORTED, launching nothing, when
// lcm(te * esize, 16) exceeds the staging buffer.
swz_status launch_staged_tiles(void *dst, const void *src, int64_t n_elems, int64_t te, int esize, int B, int M,
                               int S, int steps, cudaStream_t st) {
    const int64_t tile_bytes = te * esize;
    int64_t g = tile_bytes, h = 16;
    while (h) { const int64_t r = g % h; g = h; h = r; }
    const int64_t l = tile_bytes / g * 16;  // lcm(tile bytes, 16)
    if (l > kStageBytes) return SWZ_ERR_UNSUPPORTED;
    const int block = static_cast<int>(l * (kStageBytes / l));
    const int64_t bytes = n_elems * esize;
    const int a_src = static_cast<int>(reinterpret_cast<uintptr_t>(src) & 15u);
    const int a_dst = static_cast<int>(reinterpret_cast<uintptr_t>(dst) & 15u);
    const bool mis = (a_src | a_dst) != 0;
    // groups of 2^M elements move intact: gather units of 2^k elements,
    // k = min(M, log2(16 / esize)), under Swizzle<B, M - k, S> on unit
    // offsets (tiles hold a multiple of 2^M elements); a unit also has to
    // keep the alignment of both pointers within their 16-byte chunks
    int k = 0;
    while (k < M && (esize << (k + 1)) <= 8 && ((a_src | a_dst) % (esize << (k + 1))) == 0) ++k;
    if (te <= 0 || te % (int64_t(1) << k) != 0) return SWZ_ERR_UNSUPPORTED;  // blocks of whole units only
    const int64_t te_u = te >> k;
#define SWZ_STAGED(U) (mis ? launch_staged<U, true>(dst, src, bytes, block, te_u, B, M - k, S, steps, a_src, a_dst, st) \
                           : launch_staged<U, false>(dst, src, bytes, block, te_u, B, M - k, S, steps, 0, 0, st))
    switch (esize << k) {
        case 1: return SWZ_STAGED(1);
        case 2: return SWZ_STAGED(2);
        case 4: return SWZ_STAGED(4);
        default: return SWZ_STAGED(8);
    }
#undef SWZ_STAGED
}

// relayout_warp_coset_kernel for a negative shift whose map keeps each
// destination vector's sources inside its aligned block of 32 vectors;
// SWZ_ERR_UNSUPPORTED (nothing launched) otherwise.
swz_status launch_warp_coset(void *dst, const void *src, int64_t n_elems, int esize, int B, int M, int S, int steps,
                             cudaStream_t st) {
    int lv = 0;
    while ((1 << lv) < 16 / esize) ++lv;
    if (B <= 0 || S >= 0 || M >= lv || sw_write_hi(B, M, S) <= lv) return SWZ_ERR_UNSUPPORTED;
    const uint64_t V = 1ull << lv;
    // the smallest block (32 or 64 vectors) that Gv keeps for every vector bit
    // of a closure block, and that holds every unit's offset
    int nb = 0;
    // (64-vector blocks take two shuffles per unit: for 1-byte units, 32 per
    // vector, which ran at 0.67 of the copy bandwidth where the register
    // kernel reaches 0.92, so those stay there)
    const int max_nb = (esize << M) == 1 ? 1 : 2;
    for (int cand = 1; cand <= max_nb && nb == 0; ++cand) {
        const int shift = cand == 1 ? 5 : 6;
        bool ok = true;
        for (int b = 0; ok && b < sw_write_hi(B, M, S) - lv; ++b) {
            const uint64_t y = sw_inv((1ull << b) << lv, B, M, S, steps);
            ok = (y & (V - 1)) == 0 && ((y >> lv) >> shift) == ((1ull << b) >> shift);
        }
        const int U0 = esize << M;
        for (int t = 0; ok && t < 16 / U0; ++t)
            ok = (sw_inv(static_cast<uint64_t>(t) * (U0 / esize), B, M, S, steps) >> lv) < (32ull * cand);
        if (ok) nb = cand;
    }
    if (nb == 0) return SWZ_ERR_UNSUPPORTED;
    WarpCosetArgs a{};
    a.dst = static_cast<uint4 *>(dst);
    a.src = static_cast<const uint4 *>(src);
    a.nvec = n_elems * esize / 16;
    a.B = B; a.M = M; a.S = S;
    a.steps = steps;
    a.lv = lv;
    const int U = esize << M;
    for (int t = 0; t < 16 / U; ++t)
        a.off[t] = static_cast<uint32_t>(sw_inv(static_cast<uint64_t>(t) * (U / esize), B, M, S, steps) >> lv);
    int src_lane[16];
    bool map = false;
    for (int l = 0; l < static_cast<int>(V); ++l) {
        src_lane[l] = static_cast<int>(sw_inv(static_cast<uint64_t>(l), B, M, S, steps) & (V - 1));
        map = map || src_lane[l] != l;
    }
    lane_map_selectors(src_lane, esize, a.perm_sel);
    const int64_t wave = static_cast<int64_t>(sm_count()) * 2048;
    a.per_thread = (a.nvec >= 4 * wave) ? 4 : (a.nvec >= 2 * wave || nb == 2) ? 2 : 1;  // (even for 64-blocks)
    const int64_t per_cta = int64_t(256) * a.per_thread;
    const int64_t grid = (a.nvec + per_cta - 1) / per_cta;
    if (grid > 0x7fffffffLL) return SWZ_ERR_SHAPE;
    if (grid == 0) return SWZ_OK;
    const dim3 gr(static_cast<unsigned>(grid));
#define SWZ_W(UU, NB) (map ? launch_pdl(relayout_warp_coset_kernel<UU, true, NB>, gr, dim3(256), 0, st, a) \
                           : launch_pdl(relayout_warp_coset_kernel<UU, false, NB>, gr, dim3(256), 0, st, a))
    if (nb == 1) {
        switch (U) {
            case 1: return launched(SWZ_W(1, 1));
            case 2: return launched(SWZ_W(2, 1));
            case 4: return launched(SWZ_W(4, 1));
            // U = 8 puts the written field at or above the lanes: no lane map
            default: return launched(launch_pdl(relayout_warp_coset_kernel<8, false, 1>, gr, dim3(256), 0, st, a));
        }
    }
    switch (U) {
        case 2: return launched(SWZ_W(2, 2));
        case 4: return launched(SWZ_W(4, 2));
        default: return launched(launch_pdl(relayout_warp_coset_kernel<8, false, 2>, gr, dim3(256), 0, st, a));
    }
#undef SWZ_W
}

// relayout_coset_kernel for a negative shift with M < log2 V <= M + |S|;
// SWZ_ERR_UNSUPPORTED (nothing launched) otherwise.  The bases of W and W'
// and the pivots of W' are computed here, once per launch.
swz_status launch_coset(void *dst, const void *src, int64_t n_elems, int esize, int B, int M, int S, int steps,
                        cudaStream_t st) {
    int lv = 0;
    while ((1 << lv) < 16 / esize) ++lv;
    if (B <= 0 || S >= 0 || M >= lv || M - S < lv) return SWZ_ERR_UNSUPPORTED;
    const int g = ((M + B < lv) ? M + B : lv) - M;  // 1..4
    const int U = esize << M;                       // 1, 2, 4 or 8 bytes
    const int other = (steps == 1) ? sw_inv_steps(B, S) : 1;  // steps of G^-1
    CosetArgs a{};
    a.dst = static_cast<uint4 *>(dst);
    a.src = static_cast<const uint4 *>(src);
    const int64_t nvec = n_elems * esize / 16;
    a.n_cosets = nvec >> g;
    a.B = B; a.M = M; a.S = S;
    a.steps = steps;
    a.lv = lv;
    uint64_t r[4];
    for (int i = 0; i < g; ++i) {
        a.w[i] = sw_inv(1ull << (M + i), B, M, S, steps) >> lv;
        a.wd[i] = sw_inv(a.w[i] << lv, B, M, S, other) >> lv;
        r[i] = a.wd[i];
    }
    // reduced echelon form of W': pivot i is the top bit of row i, cleared
    // from every other row
    for (int i = 0; i < g; ++i) {
        for (int k = 0; k < i; ++k)
            if ((r[i] >> a.pivot[k]) & 1u) r[i] ^= r[k];
        if (r[i] == 0) return SWZ_ERR_UNSUPPORTED;  // (W' has dimension g for every valid swizzle)
        int p = 63;
        while (!((r[i] >> p) & 1u)) --p;
        a.pivot[i] = p;
        for (int k = 0; k < i; ++k)
            if ((r[k] >> p) & 1u) r[k] ^= r[i];
    }
    std::sort(a.pivot, a.pivot + g);
    // disjoint fields with r >= 2 read-field bits above the lanes: 2^SB cosets
    // per thread over the region bits (then W = W' is the g bits below bit |S|)
    const int r_above = B - g;
    const int sbits = (-S >= B && r_above >= 2) ? std::min(std::min(r_above, 3), 4 - g) : 0;
    if (sbits > 0) {
        a.sbase = -S - g;
        a.n_cosets = nvec >> (g + sbits);  // threads
    }
    // block stores: w'_i = e_i, destination 32-byte aligned (instantiated where
    // such cosets occur outside the warp kernel's reach: U * 2^g = 16)
    bool st32 = sbits == 0 && (U << g) == 16 && (reinterpret_cast<uintptr_t>(dst) & 31u) == 0;
    for (int i = 0; st32 && i < g; ++i) st32 = a.wd[i] == (1ull << i);
    const int nc = sbits > 0 ? 1 : (g >= 3) ? 1 : (8 >> g);
    const int64_t per_cta = int64_t(256) * nc;
    const int64_t grid = (a.n_cosets + per_cta - 1) / per_cta;
    if (grid > 0x7fffffffLL) return SWZ_ERR_SHAPE;
    if (grid == 0) return SWZ_OK;
    const dim3 gr(static_cast<unsigned>(grid));
#define SWZ_C(UU, GG, SS) launched(launch_pdl(relayout_coset_kernel<UU, GG, SS, false>, gr, dim3(256), 0, st, a))
#define SWZ_C32(UU, GG)                                                                                 \
    launched(st32 ? launch_pdl(relayout_coset_kernel<UU, GG, 0, true>, gr, dim3(256), 0, st, a)          \
                  : launch_pdl(relayout_coset_kernel<UU, GG, 0, false>, gr, dim3(256), 0, st, a))
    switch ((U * 8 + g) * 4 + sbits) {
        case (1 * 8 + 1) * 4: return SWZ_C(1, 1, 0);
        case (1 * 8 + 2) * 4: return SWZ_C(1, 2, 0);
        case (1 * 8 + 3) * 4: return SWZ_C(1, 3, 0);
        case (1 * 8 + 4) * 4: return SWZ_C32(1, 4);
        case (2 * 8 + 1) * 4: return SWZ_C(2, 1, 0);
        case (2 * 8 + 2) * 4: return SWZ_C(2, 2, 0);
        case (2 * 8 + 3) * 4: return SWZ_C32(2, 3);
        case (4 * 8 + 1) * 4: return SWZ_C(4, 1, 0);
        case (4 * 8 + 2) * 4: return SWZ_C32(4, 2);
        case (8 * 8 + 1) * 4: return SWZ_C32(8, 1);
        // (r >= 2 means g = log2 V - M, so U = 16 >> g)
        case (8 * 8 + 1) * 4 + 2: return SWZ_C(8, 1, 2);
        case (8 * 8 + 1) * 4 + 3: return SWZ_C(8, 1, 3);
        case (4 * 8 + 2) * 4 + 2: return SWZ_C(4, 2, 2);
        case (2 * 8 + 3) * 4 + 1: return SWZ_C(2, 3, 1);
        default: return SWZ_ERR_UNSUPPORTED;
    }
#undef SWZ_C32
#undef SWZ_C
}

// relayout_coset_map_kernel for a negative shift with M + |S| < log2 V <
// M + |S| + B and g <= 3; SWZ_ERR_UNSUPPORTED (nothing launched) otherwise.
swz_status launch_coset_map(void *dst, const void *src, int64_t n_elems, int esize, int B, int M, int S,
                            int steps, cudaStream_t st) {
    int lv = 0;
    while ((1 << lv) < 16 / esize) ++lv;
    if (B <= 0 || S >= 0 || M >= lv || M - S >= lv || M - S + B <= lv) return SWZ_ERR_UNSUPPORTED;
    const int V = 1 << lv;
    const int other = (steps == 1) ? sw_inv_steps(B, S) : 1;  // steps of G^-1
    CosetMapArgs a{};
    CosetArgs &c = a.c;
    c.dst = static_cast<uint4 *>(dst);
    c.src = static_cast<const uint4 *>(src);
    c.B = B; c.M = M; c.S = S;
    c.steps = steps;
    c.lv = lv;
    // images of the lane bits: lane part lam[i], vector part u[i]; a basis of
    // W from them in lane order, and the coordinates phi_bit[i] of each u[i]
    int lam[4] = {0, 0, 0, 0};
    uint32_t phi_bit[4] = {0, 0, 0, 0};
    uint64_t red[4];
    uint32_t combo[4];
    int rpiv[4];
    int g = 0;
    for (int i = 0; i < lv; ++i) {
        const uint64_t img = sw_inv(1ull << i, B, M, S, steps);
        lam[i] = static_cast<int>(img & (V - 1));
        const uint64_t u = img >> lv;
        uint64_t x = u;
        uint32_t cm = 0;
        for (int t = 0; t < g; ++t)
            if ((x >> rpiv[t]) & 1u) { x ^= red[t]; cm ^= combo[t]; }
        if (x == 0) { phi_bit[i] = cm; continue; }
        if (g == 3) return SWZ_ERR_UNSUPPORTED;  // (g = 4 does not occur in the parameter ranges)
        int p = 63;
        while (!((x >> p) & 1u)) --p;
        const uint32_t cx = cm ^ (1u << g);  // x as a combination of basis elements
        for (int k = 0; k < g; ++k)
            if ((red[k] >> p) & 1u) { red[k] ^= x; combo[k] ^= cx; }
        c.w[g] = u;
        red[g] = x; rpiv[g] = p; combo[g] = cx;
        phi_bit[i] = 1u << g;
        ++g;
    }
    if (g == 0) return SWZ_ERR_UNSUPPORTED;
    // Lam and phi on every lane; the byte permutation and the masks
    int src_lane[16];
    uint32_t phi[16];
    for (int l = 0; l < V; ++l) {
        int lm = 0;
        uint32_t ph = 0;
        for (int i = 0; i < lv; ++i)
            if ((l >> i) & 1) { lm ^= lam[i]; ph ^= phi_bit[i]; }
        src_lane[l] = lm;
        phi[l] = ph;
    }
    lane_map_selectors(src_lane, esize, a.perm_sel);
    for (int byte = 0; byte < 16; ++byte)
        a.mask[phi[byte / esize]][byte >> 2] |= 0xffu << ((byte & 3) * 8);
    // W' and its pivots
    uint64_t r[4];
    bool wd_low = true;  // W' spanned by the lowest g vector bits
    for (int i = 0; i < g; ++i) {
        const uint64_t y = sw_inv(c.w[i] << lv, B, M, S, other);
        if (y & (V - 1)) return SWZ_ERR_UNSUPPORTED;  // (G^-1 keeps lane bits of a vector offset at 0)
        c.wd[i] = y >> lv;
        r[i] = c.wd[i];
        wd_low = wd_low && c.wd[i] < (1ull << g);
    }
    bool st32 = false;
    if (wd_low) {
        // change of basis: w'_i = e_i, w_i = Gv(e_i); phi again, as coordinates
        // of each lane bit's vector image in the new w basis
        for (int i = 0; i < g; ++i) {
            c.wd[i] = 1ull << i;
            const uint64_t y = sw_inv((1ull << i) << lv, B, M, S, steps);
            if (y & (V - 1)) return SWZ_ERR_UNSUPPORTED;
            c.w[i] = y >> lv;
            r[i] = c.wd[i];
        }
        uint64_t nred[4];
        uint32_t ncombo[4];
        int npiv[4];
        for (int i = 0; i < g; ++i) {  // reduced echelon form of the new w basis
            uint64_t x = c.w[i];
            uint32_t cx = 1u << i;
            for (int t = 0; t < i; ++t)
                if ((x >> npiv[t]) & 1u) { x ^= nred[t]; cx ^= ncombo[t]; }
            if (x == 0) return SWZ_ERR_UNSUPPORTED;
            int p = 63;
            while (!((x >> p) & 1u)) --p;
            for (int t = 0; t < i; ++t)
                if ((nred[t] >> p) & 1u) { nred[t] ^= x; ncombo[t] ^= cx; }
            nred[i] = x; ncombo[i] = cx; npiv[i] = p;
        }
        for (int i = 0; i < lv; ++i) {
            uint64_t x = sw_inv(1ull << i, B, M, S, steps) >> lv;
            uint32_t cx = 0;
            for (int t = 0; t < g; ++t)
                if ((x >> npiv[t]) & 1u) { x ^= nred[t]; cx ^= ncombo[t]; }
            if (x != 0) return SWZ_ERR_UNSUPPORTED;  // (the images span W)
            phi_bit[i] = cx;
        }
        for (int l = 0; l < V; ++l) {
            uint32_t ph = 0;
            for (int i = 0; i < lv; ++i)
                if ((l >> i) & 1) ph ^= phi_bit[i];
            phi[l] = ph;
        }
        for (int m = 0; m < 8; ++m)
            for (int w = 0; w < 4; ++w) a.mask[m][w] = 0;
        for (int byte = 0; byte < 16; ++byte)
            a.mask[phi[byte / esize]][byte >> 2] |= 0xffu << ((byte & 3) * 8);
        st32 = (reinterpret_cast<uintptr_t>(dst) & 31u) == 0;
    }
    for (int i = 0; i < g; ++i) {
        for (int k = 0; k < i; ++k)
            if ((r[i] >> c.pivot[k]) & 1u) r[i] ^= r[k];
        if (r[i] == 0) return SWZ_ERR_UNSUPPORTED;
        int p = 63;
        while (!((r[i] >> p) & 1u)) --p;
        c.pivot[i] = p;
        for (int k = 0; k < i; ++k)
            if ((r[k] >> p) & 1u) r[k] ^= r[i];
    }
    std::sort(c.pivot, c.pivot + g);
    const int64_t nvec = n_elems * esize / 16;
    c.n_cosets = nvec >> g;
    const int nc = (g >= 3) ? 1 : (8 >> g);
    const int64_t per_cta = int64_t(256) * nc;
    const int64_t grid = (c.n_cosets + per_cta - 1) / per_cta;
    if (grid > 0x7fffffffLL) return SWZ_ERR_SHAPE;
    if (grid == 0) return SWZ_OK;
    const dim3 gr(static_cast<unsigned>(grid));
#define SWZ_M(GG)                                                                              \
    launched(st32 ? launch_pdl(relayout_coset_map_kernel<GG, true>, gr, dim3(256), 0, st, a)      \
                  : launch_pdl(relayout_coset_map_kernel<GG, false>, gr, dim3(256), 0, st, a))
    switch (g) {
        case 1: return SWZ_M(1);
        case 2: return SWZ_M(2);
        default: return SWZ_M(3);
    }
#undef SWZ_M
}

swz_status launch_scalar_any(void *dst, const void *src, int64_t n_elems, int64_t tile_elems, int esize, int B,
                             int M, int S, int steps, cudaStream_t st) {
    switch (esize) {
        case 1: return launch_scalar<1>(dst, src, n_elems, tile_elems, B, M, S, steps, st);
        case 2: return launch_scalar<2>(dst, src, n_elems, tile_elems, B, M, S, steps, st);
        case 4: return launch_scalar<4>(dst, src, n_elems, tile_elems, B, M, S, steps, st);
        case 8: return launch_scalar<8>(dst, src, n_elems, tile_elems, B, M, S, steps, st);
        case 16: return launch_scalar<16>(dst, src, n_elems, tile_elems, B, M, S, steps, st);
        default: return SWZ_ERR_PARAM;
    }
}

}  // namespace

// Arguments are validated by the caller (swz_relayout in swz_abi.cu).
swz_status relayout_launch(void *dst, const void *src, int64_t n_tiles, int64_t tile_elems,
                           int esize, int B, int M, int S, int direction, cudaStream_t st) {
    const int64_t n_elems = n_tiles * tile_elems;
    const int steps = direction == 0 ? sw_inv_steps(B, S) : 1;
    const int64_t tile_bytes = tile_elems * esize;
    const bool aligned16 = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
    const bool link_grid = host_resident(dst) || host_resident(src);
    int lv = 0;
    while ((1 << lv) < 16 / esize) ++lv;
    if (tile_bytes < 16 && 16 % tile_bytes == 0 && aligned16 && (n_elems * esize) % 16 == 0)
        return launch_lane_map(dst, src, n_elems, esize, static_cast<int>(tile_elems), B, M, S, steps, link_grid,
                               st);
    // Tiles holding whole swizzle periods (2^(B+M+|S|) elements) see the same
    // swizzle on whole-buffer offsets, so a buffer of whole 16-byte vectors runs
    // as one tile whatever the tile's own size.
    const int period = B + M + (S < 0 ? -S : S);  // the offset bits the swizzle touches
    if (n_tiles > 1 && tile_bytes % 16 != 0 && aligned16 && (n_elems * esize) % 16 == 0 &&
        (B == 0 || (period < 62 && tile_elems % (int64_t(1) << period) == 0)))
        return relayout_launch(dst, src, 1, n_elems, esize, B, M, S, direction, st);
    if (tile_bytes % 16 != 0 && aligned16) {
        const swz_status s = launch_staged_tiles(dst, src, n_elems, tile_elems, esize, B, M, S, steps, st);
        if (s != SWZ_ERR_UNSUPPORTED) return s;
    }
    if (B > 0 && S < 0 && M < lv && tile_bytes % 16 == 0 && aligned16) {
        // A negative shift reads the field at M, below the lane bits of a
        // vector, and writes |S| bits higher.  The offsets close under the
        // swizzle in aligned blocks of 2^wtop elements (tiles are multiples
        // of such blocks).  Blocks inside one vector: a fixed lane map.
        // Otherwise the lanes of one destination vector come from several
        // source vectors.  When they stay inside the destination's block of
        // 32 vectors, warp shuffles gather them; otherwise cosets of whole
        // vectors in registers (with a fixed lane map when the written field
        // starts inside the lanes); what none covers goes through blocks of up
        // to the staging size in shared memory, else element by element.
        const int wtop = sw_write_hi(B, M, S);
        if (wtop <= lv)
            return launch_lane_map(dst, src, n_elems, esize, 1 << wtop, B, M, S, steps, link_grid, st);
        const swz_status sw = launch_warp_coset(dst, src, n_elems, esize, B, M, S, steps, st);
        if (sw != SWZ_ERR_UNSUPPORTED) return sw;
        const swz_status sc = launch_coset(dst, src, n_elems, esize, B, M, S, steps, st);
        if (sc != SWZ_ERR_UNSUPPORTED) return sc;
        const swz_status sm = launch_coset_map(dst, src, n_elems, esize, B, M, S, steps, st);
        if (sm != SWZ_ERR_UNSUPPORTED) return sm;
        const swz_status s = launch_staged_tiles(dst, src, n_elems, int64_t(1) << wtop, esize, B, M, S, steps, st);
        if (s != SWZ_ERR_UNSUPPORTED) return s;
        return launch_scalar_any(dst, src, n_elems, tile_elems, esize, B, M, S, steps, st);
    }
    // (a negative shift with M < log2 V splits vectors: not for this kernel)
    if (tile_bytes % 16 == 0 && (aligned16 || esize < 16) && !(B > 0 && S < 0 && M < lv)) {
        RelayoutArgs a;
        a.dst = static_cast<uint4 *>(dst);
        a.src = static_cast<const uint4 *>(src);
        a.nvec = n_elems * esize / 16;
        a.tile_vecs = tile_bytes / 16;
        a.B = B; a.M = M; a.S = S;
        a.steps = steps;
        // keep each SM fed: up to four vectors per thread once the grid is
        // several waves deep (every SM x 2048 threads per wave)
        const int64_t wave = static_cast<int64_t>(sm_count()) * 2048;
        a.per_thread = (a.nvec >= 4 * wave) ? 4 : (a.nvec >= 2 * wave) ? 2 : 1;
        // kLanesGeneral: out lane l = (lanes XOR-ed by k)[L(l)], L(l) = g(l) for a lane index l
        int src_lane[16];
        for (int l = 0; l < 16 / esize; ++l)
            src_lane[l] = static_cast<int>(sw_inv(static_cast<uint64_t>(l), B, M, S, steps) & ((16 / esize) - 1));
        lane_map_selectors(src_lane, esize, a.perm_sel);
        // (a negative shift reaches here only with M >= log2 V: whole vectors move)
        const int mode = (B == 0 || M >= lv) ? kLanesFixed : (M + S >= lv) ? kLanesXor : kLanesGeneral;
        const bool local = B > 0 && (period >= 62 || (tile_elems & ((1LL << period) - 1)) != 0);
        if (!aligned16) {
            const int a_src = static_cast<int>(reinterpret_cast<uintptr_t>(src) & 15u);
            const int a_dst = static_cast<int>(reinterpret_cast<uintptr_t>(dst) & 15u);
            switch (esize) {
                case 1: return launch_vec_mis<1>(a, mode, local, a_src, a_dst, st);
                case 2: return launch_vec_mis<2>(a, mode, local, a_src, a_dst, st);
                case 4: return launch_vec_mis<4>(a, mode, local, a_src, a_dst, st);
                default: return launch_vec_mis<8>(a, mode, local, a_src, a_dst, st);
            }
        }
        switch (esize) {
            case 1: return launch_vec<1>(a, mode, local, link_grid, st);
            case 2: return launch_vec<2>(a, mode, local, link_grid, st);
            case 4: return launch_vec<4>(a, mode, local, link_grid, st);
            case 8: return launch_vec<8>(a, mode, local, link_grid, st);
            case 16: return launch_vec<16>(a, mode, local, link_grid, st);
            default: return SWZ_ERR_PARAM;
        }
    }
    if (!aligned16 && esize < 16) {
        // Pointers not 16-byte aligned: the staged kernel in its MIS form over
        // the smallest blocks the swizzle maps onto themselves (a swizzle
        // period when the tiles hold whole periods, else a tile); blocks
        // larger than the staging buffer go element by element.
        // (blocks are whole groups of 2^M elements: the gather moves units of
        // up to 2^M elements, and every tile holds whole groups)
        int64_t te_c = tile_elems;
        if (B == 0) te_c = int64_t(1) << M;
        else if (period < 62 && tile_elems % (int64_t(1) << period) == 0) te_c = int64_t(1) << period;
        const swz_status s = launch_staged_tiles(dst, src, n_elems, te_c, esize, B, M, S, steps, st);
        if (s != SWZ_ERR_UNSUPPORTED) return s;
    }
    return launch_scalar_any(dst, src, n_elems, tile_elems, esize, B, M, S, steps, st);
}

}  // namespace swz
