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
//     vectors): a fixed lane map, warp shuffles within blocks of 32 or 64
//     vectors (relayout_warp_coset_kernel), cosets of whole vectors in
//     registers (relayout_coset_kernel, relayout_coset_map_kernel; these three
//     in swz_relayout_neg.cu), the staged kernel over closure blocks, or
//     element by element;
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
    int once = 0;       // stores marked evict-first: the output is larger than L2
    uint32_t perm_sel[12];  // kLanesGeneral: prmt selectors of the fixed lane map L, 3 per word
};

constexpr int kMaxPerThread = 4;


// LINK: the variant for host-resident buffers, whose grid is sized for the
// host link: the grid walks the buffer in strides of itself, and loads carry
// no L2 eviction hint (with the evict-first hint a host-reading launch beside
// a host-writing one moved 12% less over the link).  Otherwise one CTA covers
// one stretch of blockDim.x * per_thread vectors, loads marked evict-first.
// At most 40 registers (6 CTAs per SM) with whole-buffer offsets; tile-local
// offsets need a few more (5 CTAs per SM).
template <int E, int MODE, bool LOCAL, bool LINK>
__global__ void __launch_bounds__(256, LOCAL ? 5 : 6) relayout_vec_kernel(const RelayoutArgs a) {
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
        const uint64_t store_policy = a.once ? policy : l2_evict_normal_policy();
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
                st_hint16(a.dst + u, out, store_policy);
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

// x[w] := x[(w + g) & 3] (LEFT) or x[(w - g) & 3], g in 0..3 and different
// across lanes: two conditional steps, so the words stay in registers.
template <bool LEFT>
__device__ __forceinline__ void rotate_words(uint32_t (&x)[4], int g) {
    const uint32_t a0 = x[0], a1 = x[1], a2 = x[2], a3 = x[3];
    const bool one = g & 1;
    uint32_t b0, b1, b2, b3;
    if constexpr (LEFT) {
        b0 = one ? a1 : a0; b1 = one ? a2 : a1; b2 = one ? a3 : a2; b3 = one ? a0 : a3;
    } else {
        b0 = one ? a3 : a0; b1 = one ? a0 : a1; b2 = one ? a1 : a2; b3 = one ? a2 : a3;
    }
    const bool two = g & 2;
    x[0] = two ? b2 : b0;
    x[1] = two ? b3 : b1;
    x[2] = two ? b0 : b2;
    x[3] = two ? b1 : b3;
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
    if constexpr (!MIS) {
        a_src = 0;
        (void)a_dst;  // (only the MIS form writes at the destination's offset)
    }
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
        } else if constexpr (E == 2) {
            // A vector per thread puts the lanes 16 bytes apart, so lanes l,
            // l + 8, l + 16 and l + 24 would read one bank in every 2-byte
            // gather (4-way).  Each group of 8 lanes starts instead at another
            // word of its vector (word g = lane / 8, then g + 1, ...): the four
            // groups read four different banks, and the vector is rotated back
            // before its store.  (For 4-byte units the same form measured about
            // 1% slower than the plain order.)
            const int g = (tid >> 3) & 3;
            for (int v = tid; v < nv; v += 256) {
                const int e = v * V;
                const uint32_t p = pat == 1 ? 0u : static_cast<uint32_t>(v) - __umulhi(static_cast<uint32_t>(v), pat_recip) * pat;
                const uint4 t = *reinterpret_cast<const uint4 *>(rel_s + p * 8);
                uint32_t rw[4] = {t.x, t.y, t.z, t.w};  // the two table entries of word w's elements
                rotate_words<true>(rw, g);              // rw[w] now belongs to word (w + g) & 3
                uint32_t ow[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int s0 = e + 2 * ((w + g) & 3);  // the word's first element
                    const int r0 = static_cast<int16_t>(rw[w] & 0xffffu), r1 = static_cast<int16_t>(rw[w] >> 16);
                    const uint32_t lo = *reinterpret_cast<const uint16_t *>(sa + (s0 + r0) * 2);
                    const uint32_t hi = *reinterpret_cast<const uint16_t *>(sa + (s0 + 1 + r1) * 2);
                    ow[w] = lo | (hi << 16);
                }
                rotate_words<false>(ow, g);  // ow[w] is word w again
                st_stream16(dst + b0 + 16 * v, make_uint4(ow[0], ow[1], ow[2], ow[3]));
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
    a.once = !link_grid && n_elems * esize > l2_bytes();  // as in relayout_launch
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

// Negative shifts that split 16-byte vectors (swz_relayout_neg.cu): each
// returns SWZ_ERR_UNSUPPORTED, launching nothing, for a request outside its
// kernel's reach.
swz_status launch_warp_coset(void *dst, const void *src, int64_t n_elems, int esize, int B, int M, int S, int steps,
                             cudaStream_t st);
swz_status launch_coset(void *dst, const void *src, int64_t n_elems, int esize, int B, int M, int S, int steps,
                        cudaStream_t st);
swz_status launch_coset_map(void *dst, const void *src, int64_t n_elems, int esize, int B, int M, int S,
                            int steps, cudaStream_t st);

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
        // An output larger than L2 cannot stay there for a following launch:
        // stores marked evict-first (1 GiB: 1.042 -> 1.048 of the copy
        // bandwidth).  A smaller one keeps the default priority, so the next
        // launch finds it in L2 (evict-first stores took a 64 MiB forward +
        // inverse from 37.5 to 47.7 us).  Host-resident buffers keep it too.
        a.once = !link_grid && n_elems * esize > l2_bytes();
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
