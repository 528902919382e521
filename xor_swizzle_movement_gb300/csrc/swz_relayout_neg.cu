// swz_relayout_neg.cu -- relayouts under negative shifts whose read field
// starts below a 16-byte vector's lane bits, so a destination vector gathers
// lanes from several source vectors (sm_103a).  relayout_launch
// (swz_relayout.cu) routes such requests here, in this order: warp shuffles
// within aligned blocks of 32 or 64 vectors, then cosets of whole vectors in
// registers (with a fixed lane map when the written field starts inside the
// lanes).
#include "swz_common.cuh"

#include <algorithm>

namespace swz {
namespace {

constexpr int kMaxPerThread = 4;  // vectors in flight per thread

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

}  // namespace

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

}  // namespace swz
