// swz_transpose.cu -- HBM -> shared memory -> HBM transpose with the tile
// staged under a per-element-size swizzle (sm_103a).
//
// Every kernel fills the shared tile row-wise (coalesced 16-byte global
// loads) and drains it column-wise (coalesced 16-byte global stores of the
// transposed rows).  The column-wise drain is where a plain row-major tile
// serialises: all rows of one column sit in one bank ("CuTe Swizzle 学习手册",
// section "冲突的典型场景").  The variants differ only in where element
// (row, col) of a tile lives in shared memory:
//   SWZ_T_SWIZZLED    the column index is XOR-ed with the row index (the
//                     swizzle of the element size, below);
//   SWZ_T_UNSWIZZLED  plain [T][T];
//   SWZ_T_PADDED      [T][T + 1] ("CUDA 013 - Swizzle 的工作原理", section
//                     "如何避免 Bank Conflict").
//
// Element sizes 4 and 8: units of N x N elements with 128-byte rows (N = 32
// for 4 bytes, 16 for 8 bytes) under element Swizzle<log2 N, 0, log2 N>, i.e.
// physical column = column ^ row inside a unit ("CUDA 013 - Swizzle 的工作原理",
// sections "swizzle 映射案例" and "行列位数": 32 x 32 units for 4-byte
// elements, 16 x 16 for 8-byte ones).  Shared accesses are per element; with
// the thread mapping below, each warp-wide store touches 4 rows x one unit
// width and each warp-wide load 4 columns x one unit height, and the XOR
// spreads both over all 32 banks.  A CTA of 256 threads owns 2 x 2 units:
// 64 x 64 fp32 (16 KiB, at most 6 CTAs per SM so that no register spills) or
// 32 x 32 fp64 (8 KiB, 8 CTAs per SM: the 64 x 64 fp64 tile's 32 KiB held
// occupancy down and ran 17% slower).
//
// Element size 2: tiles of 64 x 64 with 128-byte rows under the
// byte-address Swizzle<3,4,3> (16-byte chunk index XOR row mod 8, equal to
// element Swizzle<3,3,3>; "CuTe Swizzle 学习手册", sections "Sw<3,4,3> vs
// Sw<3,3,3>" and "不同矩阵配置的选择指南").  The tile is filled with 16-byte
// stores and drained with transposing 8 x 8 matrix loads (ldmatrix .trans):
// the eight rows of one 8 x 8 block are read from eight different chunk
// positions, so each matrix load is one conflict-free pass.  Four lanes then
// exchange 32-bit words (a two-step XOR butterfly) so that each lane owns 16
// contiguous output bytes.
//
// Element size 1: tiles of 128 x 128 bytes with 128-byte rows under the
// byte-address Swizzle<3,4,7> (16-byte chunk index XOR (row / 16) mod 8).
// The tile is filled with 16-byte stores; each thread of the drain reads one
// 32-bit word (4 columns) from 16 consecutive rows, transposes the 4 x 4 byte
// blocks in registers with byte permutes and stores 4 output vectors of 16
// bytes.  A warp's drain load covers 8 row groups x 4 words, which the XOR
// spreads over all 32 banks.  The unswizzled and padded stagings of 1-byte
// elements, and the 16-byte elements, use 32 x 32 units under element
// Swizzle<5,0,5>, one element per access.
//
// Tiles that cross the matrix edge, and matrices whose rows are not whole
// 16-byte vectors, go element by element with bounds checks through the same
// shared layout.
#include "swz_common.cuh"

#include <cstring>

namespace swz {

// A transpose can hand its output straight to a forward relayout: the
// transposed matrix, cut into tiles of `te` consecutive elements, each tile
// stored in Swizzle<B,M,S> order.  Transposed element y then lands at
// fused_pos(y).  For S > 0 a 16-byte vector of it lands in one 16-byte vector
// (the swizzle only reads bits above the bits it writes), with its lanes moved
// by the inverse lane map L^-1 (fixed, `sel`) and then XOR-ed by the vector's
// k.  A negative shift reads below the bits it writes: vectors stay whole only
// when M >= log2 V; otherwise (vec_whole = 0) every element is stored on its
// own through the kernels' element path.
struct FuseArgs {
    int64_t te;         // relayout tile, elements
    int B, M, S;
    int global;         // te is a multiple of 2^(B+M+|S|): the whole-matrix offset may be swizzled directly
    int lanes;          // 0: lanes stay (M >= log2 V); 1: lanes XOR-ed by k only (M + S >= log2 V); 2: general
    int vec_whole;      // 16-byte vectors of the transposed matrix land whole
    uint32_t sel[12];   // bytes_permute selectors of L^-1, L(l) = sw(l) mod V
};

namespace {

__device__ __forceinline__ uint64_t fused_pos(uint64_t y, const FuseArgs &f) {
    if (f.global) return sw_fwd(y, f.B, f.M, f.S);
    const uint64_t loc = y % static_cast<uint64_t>(f.te);
    return (y - loc) + sw_fwd(loc, f.B, f.M, f.S);
}

template <int E>
__device__ __forceinline__ void store16_fused(void *dst, uint64_t y, uint4 v, const FuseArgs &f) {
    constexpr uint64_t VM = VecTraits<E>::V - 1;
    const uint64_t x = fused_pos(y, f);
    uint4 o = v;  // f.lanes is uniform over the launch: no divergence
    if (f.lanes == 2) o = bytes_permute(o, f.sel);
    if (f.lanes != 0) o = lanes_xor<E>(o, static_cast<uint32_t>(x & VM));
    st_stream16(static_cast<uint8_t *>(dst) + (x & ~VM) * E, o);
}

// ---------------------------------------------------------------- 4 / 8 B --
template <typename T, int VARIANT, int UR, int UC, int THREADS, int MIN_CTAS, bool FUSE>
__global__ void __launch_bounds__(THREADS, MIN_CTAS)
    transpose_unit_kernel(T *__restrict__ dst, const T *__restrict__ src, int64_t R, int64_t C,
                          int64_t tiles_c, int vec_ok, const FuseArgs f) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    constexpr int N = 128 / static_cast<int>(sizeof(T));    // unit edge: 32 (4 B) or 16 (8 B)
    constexpr int VPE = 16 / static_cast<int>(sizeof(T));   // elements per 16-byte vector
    constexpr int P = (VARIANT == SWZ_T_PADDED) ? N + 1 : N;  // unit row pitch, elements
    constexpr int TR = UR * N, TC = UC * N;                 // tile edge, elements
    constexpr int NV = TR * TC / VPE;                       // 16-byte vectors per tile
    constexpr int ITER = NV / THREADS;
    static_assert(NV % THREADS == 0, "tile must divide evenly over the threads");
    static_assert(8 * VPE == N, "a unit row is eight 16-byte vectors");
    __shared__ T sm[UR * UC * N * P];

    const int64_t tr = static_cast<int64_t>(blockIdx.x) / tiles_c;
    const int64_t tc = static_cast<int64_t>(blockIdx.x) - tr * tiles_c;
    const int64_t r0 = tr * TR, c0 = tc * TC;
    const int tid = threadIdx.x;
    auto phys = [](int ir, int ic) -> int { return VARIANT == SWZ_T_SWIZZLED ? (ic ^ ir) : ic; };

    if (vec_ok && r0 + TR <= R && c0 + TC <= C) {
        uint4 v[ITER];
        // fill: a warp covers 4 tile rows x one unit width (8 vectors per row)
#pragma unroll
        for (int k = 0; k < ITER; ++k) {
            const int id = k * THREADS + tid;
            const int lane = id & 31, wb = id >> 5;
            const int q = lane & 7, row = (wb / UC) * 4 + (lane >> 3), uc = wb % UC;
            v[k] = ld_stream16(src + (r0 + row) * C + c0 + uc * N + q * VPE);
        }
#pragma unroll
        for (int k = 0; k < ITER; ++k) {
            const int id = k * THREADS + tid;
            const int lane = id & 31, wb = id >> 5;
            const int q = lane & 7, row = (wb / UC) * 4 + (lane >> 3), uc = wb % UC;
            const int ur = row / N, ir = row % N;
            T e[VPE];
            memcpy(e, &v[k], 16);
            T *unit = sm + (ur * UC + uc) * N * P + ir * P;
#pragma unroll
            for (int j = 0; j < VPE; ++j) unit[phys(ir, q * VPE + j)] = e[j];
        }
        __syncthreads();
        // drain: a warp covers 4 output rows (tile columns) x one unit height
#pragma unroll
        for (int k = 0; k < ITER; ++k) {
            const int id = k * THREADS + tid;
            const int lane = id & 31, wb = id >> 5;
            const int p = lane & 7, ocl = (wb / UR) * 4 + (lane >> 3), ur = wb % UR;
            const int uc = ocl / N, ic = ocl % N;
            const T *unit = sm + (ur * UC + uc) * N * P;
            T e[VPE];
#pragma unroll
            for (int j = 0; j < VPE; ++j) {
                const int ir = p * VPE + j;
                e[j] = unit[ir * P + phys(ir, ic)];
            }
            uint4 o;
            memcpy(&o, e, 16);
            const int64_t y = (c0 + ocl) * R + r0 + ur * N + p * VPE;
            if constexpr (FUSE) store16_fused<static_cast<int>(sizeof(T))>(dst, static_cast<uint64_t>(y), o, f);
            else if constexpr (sizeof(T) == 8) st_once16(dst + y, o);  // streaming: 0.96 -> 1.00 of HBM on fp64 8192^2
            else st_stream16(dst + y, o);  // (streaming stores measured 0.6% slower for 4-byte elements)
        }
    } else {
        // all loads first: each thread keeps its elements of the tile in flight
        constexpr int EI = TR * TC / THREADS;
        T ev[EI];
#pragma unroll
        for (int k = 0; k < EI; ++k) {
            const int idx = k * THREADS + tid, row = idx / TC, cl = idx % TC;
            if (r0 + row < R && c0 + cl < C) ev[k] = src[(r0 + row) * C + c0 + cl];
        }
#pragma unroll
        for (int k = 0; k < EI; ++k) {
            const int idx = k * THREADS + tid, row = idx / TC, cl = idx % TC;
            if (r0 + row < R && c0 + cl < C) {
                const int ur = row / N, ir = row % N, uc = cl / N, ic = cl % N;
                sm[(ur * UC + uc) * N * P + ir * P + phys(ir, ic)] = ev[k];
            }
        }
        __syncthreads();
        for (int idx = tid; idx < TR * TC; idx += THREADS) {
            const int ocl = idx / TR, orow = idx % TR;
            if (c0 + ocl < C && r0 + orow < R) {
                const int ur = orow / N, ir = orow % N, uc = ocl / N, ic = ocl % N;
                const int64_t y = (c0 + ocl) * R + r0 + orow;
                dst[FUSE ? static_cast<int64_t>(fused_pos(static_cast<uint64_t>(y), f)) : y] =
                    sm[(ur * UC + uc) * N * P + ir * P + phys(ir, ic)];
            }
        }
    }
}

// ------------------------------------------------------------------- 2 B --
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &d0, uint32_t &d1,
                                                  uint32_t &d2, uint32_t &d3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(addr));
}

// 4 x 4 transpose of 32-bit words across the 4 lanes of a group (lane kk
// holds row kk on entry, column kk on exit): an XOR butterfly, first swapping
// 2 x 2 blocks with the lane 2 away, then single words with the neighbour.
__device__ __forceinline__ void transpose4_lanes(uint32_t &x0, uint32_t &x1, uint32_t &x2, uint32_t &x3, int kk) {
    const bool hi2 = kk & 2;
    uint32_t s0 = hi2 ? x0 : x2, s1 = hi2 ? x1 : x3;
    s0 = __shfl_xor_sync(kFullMask, s0, 2);
    s1 = __shfl_xor_sync(kFullMask, s1, 2);
    if (hi2) { x0 = s0; x1 = s1; } else { x2 = s0; x3 = s1; }
    const bool hi1 = kk & 1;
    uint32_t t0 = hi1 ? x0 : x1, t1 = hi1 ? x2 : x3;
    t0 = __shfl_xor_sync(kFullMask, t0, 1);
    t1 = __shfl_xor_sync(kFullMask, t1, 1);
    if (hi1) { x0 = t0; x2 = t1; } else { x1 = t0; x3 = t1; }
}

// Tile 64 x 64 of 16-bit elements, 128 threads.
template <int VARIANT, bool FUSE>
__global__ void __launch_bounds__(128)
    transpose16_kernel(uint16_t *__restrict__ dst, const uint16_t *__restrict__ src, int64_t R,
                       int64_t C, int64_t tiles_c, int vec_ok, const FuseArgs f) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    constexpr int TR = 64, TC = 64, THREADS = 128;
    constexpr int PITCH = (VARIANT == SWZ_T_PADDED) ? 72 : 64;  // elements per shared row
    __shared__ __align__(1024) uint16_t sm[TR * PITCH];
    const int64_t tr = static_cast<int64_t>(blockIdx.x) / tiles_c;
    const int64_t tc = static_cast<int64_t>(blockIdx.x) - tr * tiles_c;
    const int64_t r0 = tr * TR, c0 = tc * TC;
    const int tid = threadIdx.x;
    // 16-byte chunk position of chunk ch of tile row `row`
    auto chunk = [](int row, int ch) -> int { return VARIANT == SWZ_T_SWIZZLED ? (ch ^ (row & 7)) : ch; };

    if (vec_ok && r0 + TR <= R && c0 + TC <= C) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int id = k * THREADS + tid, ch = id & 7, row = id >> 3;
            v[k] = ld_stream16(src + (r0 + row) * C + c0 + ch * 8);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int id = k * THREADS + tid, ch = id & 7, row = id >> 3;
            *reinterpret_cast<uint4 *>(sm + row * PITCH + chunk(row, ch) * 8) = v[k];
        }
        __syncthreads();
        const int lane = tid & 31, warp = tid >> 5;
        const int g = lane >> 2, kk = lane & 3;   // output row in the block, word slot
        const int m = lane >> 3, i = lane & 7;    // matrix addressed by this lane, its row
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int xi = warp * 4 + k;          // 16 x4 loads cover the 64 blocks
            const int cb = xi & 7, rbg = (xi >> 3) * 4;
            const int row = (rbg + m) * 8 + i;
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4_trans(smem_u32(sm + row * PITCH + chunk(row, cb) * 8), a0, a1, a2, a3);
            // a[mm] holds output row 8cb + g, columns 8(rbg + mm) + 2kk .. +1.
            // 4 x 4 word transpose across lanes 4g .. 4g + 3: lane kk collects
            // words for columns 8(rbg + kk) .. +7.
            uint32_t b0 = a0, b1 = a1, b2 = a2, b3 = a3;
            transpose4_lanes(b0, b1, b2, b3, kk);
            const int64_t y = (c0 + cb * 8 + g) * R + r0 + (rbg + kk) * 8;
            if constexpr (FUSE) store16_fused<2>(dst, static_cast<uint64_t>(y), make_uint4(b0, b1, b2, b3), f);
            else st_stream16(dst + y, make_uint4(b0, b1, b2, b3));
        }
    } else {
        for (int idx = tid; idx < TR * TC; idx += THREADS) {
            const int row = idx / TC, cl = idx % TC;
            if (r0 + row < R && c0 + cl < C)
                sm[row * PITCH + chunk(row, cl >> 3) * 8 + (cl & 7)] = src[(r0 + row) * C + c0 + cl];
        }
        __syncthreads();
        for (int idx = tid; idx < TR * TC; idx += THREADS) {
            const int ocl = idx / TR, orow = idx % TR;
            if (c0 + ocl < C && r0 + orow < R) {
                const int64_t y = (c0 + ocl) * R + r0 + orow;
                dst[FUSE ? static_cast<int64_t>(fused_pos(static_cast<uint64_t>(y), f)) : y] =
                    sm[orow * PITCH + chunk(orow, ocl >> 3) * 8 + (ocl & 7)];
            }
        }
    }
}

// --------------------------------------------------------------------- 1 B --
// 4 x 4 byte transpose: row k of the block is w[k]; on return t[j] holds
// column j (byte k of t[j] is byte j of w[k]).
__device__ __forceinline__ void transpose4x4_bytes(const uint32_t w[4], uint32_t t[4]) {
    const uint32_t a = __byte_perm(w[0], w[1], 0x5140), b = __byte_perm(w[0], w[1], 0x7362);
    const uint32_t c = __byte_perm(w[2], w[3], 0x5140), d = __byte_perm(w[2], w[3], 0x7362);
    t[0] = __byte_perm(a, c, 0x5410);
    t[1] = __byte_perm(a, c, 0x7632);
    t[2] = __byte_perm(b, d, 0x5410);
    t[3] = __byte_perm(b, d, 0x7632);
}

// Tile 128 x 128 bytes, 256 threads.
template <bool FUSE>
__global__ void __launch_bounds__(256)
    transpose8_kernel(uint8_t *__restrict__ dst, const uint8_t *__restrict__ src, int64_t R, int64_t C,
                      int64_t tiles_c, int vec_ok, const FuseArgs f) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    constexpr int T = 128, THREADS = 256;
    __shared__ __align__(16) uint8_t sm[T * T];
    const int64_t tr = static_cast<int64_t>(blockIdx.x) / tiles_c;
    const int64_t tc = static_cast<int64_t>(blockIdx.x) - tr * tiles_c;
    const int64_t r0 = tr * T, c0 = tc * T;
    const int tid = threadIdx.x;
    // byte offset of (row, col) in the staged tile
    auto at = [](int row, int col) -> int { return row * T + ((((col >> 4) ^ (row >> 4)) & 7) << 4) + (col & 15); };

    if (vec_ok && r0 + T <= R && c0 + T <= C) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int id = k * THREADS + tid, row = id >> 3, ch = id & 7;
            v[k] = ld_stream16(src + (r0 + row) * C + c0 + ch * 16);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int id = k * THREADS + tid, row = id >> 3, ch = id & 7;
            *reinterpret_cast<uint4 *>(sm + at(row, ch * 16)) = v[k];
        }
        __syncthreads();
        // thread: word q (columns 4q .. 4q + 3) of rows 16g .. 16g + 15
        const int lane = tid & 31, warp = tid >> 5;
        const int g = lane & 7, q = 4 * warp + (lane >> 3);
        uint32_t col[4][4];  // col[j][a]: column 4q + j, rows 16g + 4a .. + 3
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            uint32_t w[4], t[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int row = 16 * g + 4 * a + k;
                w[k] = *reinterpret_cast<const uint32_t *>(sm + at(row, 4 * q));
            }
            transpose4x4_bytes(w, t);
#pragma unroll
            for (int j = 0; j < 4; ++j) col[j][a] = t[j];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t y = (c0 + 4 * q + j) * R + r0 + 16 * g;
            const uint4 o = make_uint4(col[j][0], col[j][1], col[j][2], col[j][3]);
            if constexpr (FUSE) store16_fused<1>(dst, static_cast<uint64_t>(y), o, f);
            else st_stream16(dst + y, o);
        }
    } else {
        for (int idx = tid; idx < T * T; idx += THREADS) {
            const int row = idx / T, cl = idx % T;
            if (r0 + row < R && c0 + cl < C) sm[at(row, cl)] = src[(r0 + row) * C + c0 + cl];
        }
        __syncthreads();
        for (int idx = tid; idx < T * T; idx += THREADS) {
            const int ocl = idx / T, orow = idx % T;
            if (c0 + ocl < C && r0 + orow < R) {
                const int64_t y = (c0 + ocl) * R + r0 + orow;
                dst[FUSE ? static_cast<int64_t>(fused_pos(static_cast<uint64_t>(y), f)) : y] = sm[at(orow, ocl)];
            }
        }
    }
}

// --------------------------------------------------------------- 1 / 16 B --
template <typename T, int VARIANT, bool FUSE>
__global__ void __launch_bounds__(256)
    transpose_generic_kernel(T *__restrict__ dst, const T *__restrict__ src, int64_t R, int64_t C,
                             int64_t tiles_c, const FuseArgs f) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    constexpr int N = 32, P = (VARIANT == SWZ_T_PADDED) ? N + 1 : N;
    __shared__ T sm[N * P];
    const int64_t tr = static_cast<int64_t>(blockIdx.x) / tiles_c;
    const int64_t tc = static_cast<int64_t>(blockIdx.x) - tr * tiles_c;
    const int64_t r0 = tr * N, c0 = tc * N;
    auto phys = [](int ir, int ic) -> int { return VARIANT == SWZ_T_SWIZZLED ? (ic ^ ir) : ic; };
    // all loads first: each thread keeps its elements of the tile in flight
    constexpr int EI = N * N / 256;
    T ev[EI];
#pragma unroll
    for (int k = 0; k < EI; ++k) {
        const int idx = k * 256 + threadIdx.x, row = idx >> 5, cl = idx & 31;
        if (r0 + row < R && c0 + cl < C) ev[k] = src[(r0 + row) * C + c0 + cl];
    }
#pragma unroll
    for (int k = 0; k < EI; ++k) {
        const int idx = k * 256 + threadIdx.x, row = idx >> 5, cl = idx & 31;
        if (r0 + row < R && c0 + cl < C) sm[row * P + phys(row, cl)] = ev[k];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < N * N; idx += 256) {
        const int ocl = idx >> 5, orow = idx & 31;
        if (c0 + ocl < C && r0 + orow < R) {
            const int64_t y = (c0 + ocl) * R + r0 + orow;
            dst[FUSE ? static_cast<int64_t>(fused_pos(static_cast<uint64_t>(y), f)) : y] = sm[orow * P + phys(orow, ocl)];
        }
    }
}

template <typename T, int UR, int UC, int THREADS, int MIN_CTAS>
swz_status launch_unit(void *dst, const void *src, int64_t R, int64_t C, int variant, bool aligned16,
                       const FuseArgs *fuse, cudaStream_t st) {
    constexpr int N = 128 / static_cast<int>(sizeof(T));
    constexpr int VPE = 16 / static_cast<int>(sizeof(T));
    const int64_t TR = UR * N, TC = UC * N;
    const int64_t tiles_c = (C + TC - 1) / TC, tiles = ((R + TR - 1) / TR) * tiles_c;
    if (tiles > 0x7fffffffLL) return SWZ_ERR_SHAPE;
    // a fused relayout needs its tiles to hold whole 16-byte vectors
    const int vec_ok = aligned16 && (C % VPE == 0) && (R % VPE == 0) && (!fuse || (fuse->te % VPE == 0 && fuse->vec_whole));
    T *d = static_cast<T *>(dst);
    const T *s = static_cast<const T *>(src);
    const unsigned g = static_cast<unsigned>(tiles);
    const FuseArgs f = fuse ? *fuse : FuseArgs{};
    cudaError_t e;
    if (fuse)
        e = launch_pdl(transpose_unit_kernel<T, SWZ_T_SWIZZLED, UR, UC, THREADS, MIN_CTAS, true>, g, dim3(THREADS), 0, st, d, s, R, C, tiles_c, vec_ok, f);
    else if (variant == SWZ_T_SWIZZLED)
        e = launch_pdl(transpose_unit_kernel<T, SWZ_T_SWIZZLED, UR, UC, THREADS, MIN_CTAS, false>, g, dim3(THREADS), 0, st, d, s, R, C, tiles_c, vec_ok, f);
    else if (variant == SWZ_T_UNSWIZZLED)
        e = launch_pdl(transpose_unit_kernel<T, SWZ_T_UNSWIZZLED, UR, UC, THREADS, MIN_CTAS, false>, g, dim3(THREADS), 0, st, d, s, R, C, tiles_c, vec_ok, f);
    else
        e = launch_pdl(transpose_unit_kernel<T, SWZ_T_PADDED, UR, UC, THREADS, MIN_CTAS, false>, g, dim3(THREADS), 0, st, d, s, R, C, tiles_c, vec_ok, f);
    return launched(e);
}

swz_status launch_16(void *dst, const void *src, int64_t R, int64_t C, int variant, bool aligned16,
                     const FuseArgs *fuse, cudaStream_t st) {
    const int64_t tiles_c = (C + 63) / 64, tiles = ((R + 63) / 64) * tiles_c;
    if (tiles > 0x7fffffffLL) return SWZ_ERR_SHAPE;
    const int vec_ok = aligned16 && (C % 8 == 0) && (R % 8 == 0) && (!fuse || (fuse->te % 8 == 0 && fuse->vec_whole));
    uint16_t *d = static_cast<uint16_t *>(dst);
    const uint16_t *s = static_cast<const uint16_t *>(src);
    const unsigned g = static_cast<unsigned>(tiles);
    const FuseArgs f = fuse ? *fuse : FuseArgs{};
    cudaError_t e;
    if (fuse)
        e = launch_pdl(transpose16_kernel<SWZ_T_SWIZZLED, true>, g, dim3(128), 0, st, d, s, R, C, tiles_c, vec_ok, f);
    else if (variant == SWZ_T_SWIZZLED)
        e = launch_pdl(transpose16_kernel<SWZ_T_SWIZZLED, false>, g, dim3(128), 0, st, d, s, R, C, tiles_c, vec_ok, f);
    else if (variant == SWZ_T_UNSWIZZLED)
        e = launch_pdl(transpose16_kernel<SWZ_T_UNSWIZZLED, false>, g, dim3(128), 0, st, d, s, R, C, tiles_c, vec_ok, f);
    else
        e = launch_pdl(transpose16_kernel<SWZ_T_PADDED, false>, g, dim3(128), 0, st, d, s, R, C, tiles_c, vec_ok, f);
    return launched(e);
}

swz_status launch_8(void *dst, const void *src, int64_t R, int64_t C, bool aligned16, const FuseArgs *fuse,
                    cudaStream_t st) {
    const int64_t tiles_c = (C + 127) / 128, tiles = ((R + 127) / 128) * tiles_c;
    if (tiles > 0x7fffffffLL) return SWZ_ERR_SHAPE;
    const int vec_ok = aligned16 && (C % 16 == 0) && (R % 16 == 0) && (!fuse || (fuse->te % 16 == 0 && fuse->vec_whole));
    uint8_t *d = static_cast<uint8_t *>(dst);
    const uint8_t *s = static_cast<const uint8_t *>(src);
    const unsigned g = static_cast<unsigned>(tiles);
    const FuseArgs f = fuse ? *fuse : FuseArgs{};
    cudaError_t e;
    if (fuse) e = launch_pdl(transpose8_kernel<true>, g, dim3(256), 0, st, d, s, R, C, tiles_c, vec_ok, f);
    else e = launch_pdl(transpose8_kernel<false>, g, dim3(256), 0, st, d, s, R, C, tiles_c, vec_ok, f);
    return launched(e);
}

template <typename T>
swz_status launch_generic(void *dst, const void *src, int64_t R, int64_t C, int variant, const FuseArgs *fuse,
                          cudaStream_t st) {
    const int64_t tiles_c = (C + 31) / 32, tiles = ((R + 31) / 32) * tiles_c;
    if (tiles > 0x7fffffffLL) return SWZ_ERR_SHAPE;
    T *d = static_cast<T *>(dst);
    const T *s = static_cast<const T *>(src);
    const unsigned g = static_cast<unsigned>(tiles);
    const FuseArgs f = fuse ? *fuse : FuseArgs{};
    cudaError_t e;
    if (fuse)
        e = launch_pdl(transpose_generic_kernel<T, SWZ_T_SWIZZLED, true>, g, dim3(256), 0, st, d, s, R, C, tiles_c, f);
    else if (variant == SWZ_T_SWIZZLED)
        e = launch_pdl(transpose_generic_kernel<T, SWZ_T_SWIZZLED, false>, g, dim3(256), 0, st, d, s, R, C, tiles_c, f);
    else if (variant == SWZ_T_UNSWIZZLED)
        e = launch_pdl(transpose_generic_kernel<T, SWZ_T_UNSWIZZLED, false>, g, dim3(256), 0, st, d, s, R, C, tiles_c, f);
    else
        e = launch_pdl(transpose_generic_kernel<T, SWZ_T_PADDED, false>, g, dim3(256), 0, st, d, s, R, C, tiles_c, f);
    return launched(e);
}

swz_status dispatch(void *dst, const void *src, int64_t R, int64_t C, int esize, int variant, const FuseArgs *fuse,
                    cudaStream_t st);

}  // namespace

swz_status transpose_tma_launch(void *dst, const void *src, int64_t R, int64_t C, cudaStream_t st);

namespace {
swz_status dispatch(void *dst, const void *src, int64_t R, int64_t C, int esize, int variant, const FuseArgs *fuse,
                    cudaStream_t st) {
    const bool aligned16 = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
    switch (esize) {
        case 1:
            if (fuse || variant == SWZ_T_SWIZZLED) return launch_8(dst, src, R, C, aligned16, fuse, st);
            return launch_generic<uint8_t>(dst, src, R, C, variant, fuse, st);
        case 2:
            if (variant == SWZ_T_TMA && !fuse) return transpose_tma_launch(dst, src, R, C, st);
            return launch_16(dst, src, R, C, variant, aligned16, fuse, st);
        case 4: return launch_unit<uint32_t, 2, 2, 256, 6>(dst, src, R, C, variant, aligned16, fuse, st);
        case 8: return launch_unit<unsigned long long, 2, 2, 256, 8>(dst, src, R, C, variant, aligned16, fuse, st);
        case 16: return launch_generic<uint4>(dst, src, R, C, variant, fuse, st);
        default: return SWZ_ERR_PARAM;
    }
}
}  // namespace

// Arguments are validated by the caller (swz_transpose in swz_abi.cu).
swz_status transpose_launch(void *dst, const void *src, int64_t R, int64_t C, int esize, int variant,
                            cudaStream_t st) {
    return dispatch(dst, src, R, C, esize, variant, nullptr, st);
}

// Arguments are validated by the caller (swz_transpose_relayout in swz_abi.cu).
swz_status transpose_relayout_launch(void *dst, const void *src, int64_t R, int64_t C, int esize, int64_t te,
                                     int B, int M, int S, cudaStream_t st) {
    FuseArgs f{};
    f.te = te;
    f.B = B;
    f.M = M;
    f.S = S;
    const int period = B + M + (S < 0 ? -S : S);  // the offset bits the swizzle touches
    f.global = (B == 0) || (period < 62 && te % (int64_t(1) << period) == 0);
    // L(l) = sw(l) mod V on the lanes of a 16-byte vector; bytes_permute needs L^-1
    const int lanes = 16 / esize;
    int L[16], Linv[16];
    for (int l = 0; l < lanes; ++l) L[l] = static_cast<int>(sw_fwd(static_cast<uint64_t>(l), B, M, S) & (lanes - 1));
    for (int l = 0; l < lanes; ++l) Linv[L[l]] = l;
    lane_map_selectors(Linv, esize, f.sel);
    int lv = 0;
    while ((1 << lv) < lanes) ++lv;
    f.lanes = (B == 0 || M >= lv) ? 0 : (M + S >= lv) ? 1 : 2;
    f.vec_whole = (B == 0 || S > 0 || M >= lv) ? 1 : 0;
    return dispatch(dst, src, R, C, esize, SWZ_T_SWIZZLED, &f, st);
}

}  // namespace swz
