// swz_probe.cu -- shared-memory staging probe (sm_103a): a diagnostic that
// repeats the fill and drain accesses of one transpose staging on register
// data, so that ncu's shared-memory bank-conflict counters can be read on the
// staging alone.
//
// Each CTA owns one shared tile laid out exactly as the transpose kernel of
// that element size and variant lays it out, and each thread issues the same
// shared-memory instructions at the same addresses as that kernel's fill
// (row-wise stores) and drain (column-wise loads):
//   4 / 8 bytes: 2 x 2 units of N x N elements (N = 128 / element size),
//                element Swizzle<log2 N, 0, log2 N>, [N][N] or [N][N + 1];
//   2 bytes:     64 x 64 with 16-byte chunk c of row r at c ^ (r mod 8)
//                (byte-address Swizzle<3,4,3>), plain, or rows of 72
//                elements; the drain reads with ldmatrix .x4 .trans;
//                SWZ_T_TMA adds the TMA kernel's second tile: each drained
//                8 x 8 block is written with stmatrix .x4 into an output
//                tile under the same swizzle (which the tensor store reads
//                in the transpose; here nothing reads it);
//   1 byte:      128 x 128 bytes, 16-byte chunk c of row r at
//                c ^ ((r / 16) mod 8) (byte-address Swizzle<3,4,7>).
// A tile is filled and drained `iters` times.  With no global buffer given the
// kernel touches no global memory at all, so every shared-memory wavefront
// the counters see belongs to the staging.  With a global source (and
// destination) buffer, each iteration also streams 16-byte vectors through it
// as the transpose does (its loads before the fill, its stores after the
// drain), which isolates the effect of concurrent global traffic on the same
// counters.
#include "swz_common.cuh"

#include <cstring>

namespace swz {
namespace {

struct ProbeArgs {
    const uint4 *gsrc;  // optional: streamed 16-byte loads, one per fill vector
    uint4 *gdst;        // optional: streamed 16-byte stores, one per drain vector
    int64_t gvecs;      // 16-byte vectors in gsrc / gdst
    int iters;
    uint32_t *sink;     // optional: one word per CTA, written after the loop
};

__device__ __forceinline__ void probe_ldmatrix_x4_trans(uint32_t addr, uint32_t &d0, uint32_t &d1, uint32_t &d2,
                                                        uint32_t &d3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ uint32_t fold(uint4 v) { return v.x ^ v.y ^ v.z ^ v.w; }

// Streamed global traffic of one iteration: vector k of thread `g` in round `it`.
__device__ __forceinline__ int64_t probe_gvec(const ProbeArgs &a, int it, int k, int per_thread) {
    const int64_t total = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    return ((static_cast<int64_t>(it) * per_thread + k) * total + g) % a.gvecs;
}

// ------------------------------------------------------------- 4 / 8 bytes --
// The unit staging of the 4- and 8-byte transpose: 256 threads, 2 x 2 units.
template <typename T, int VARIANT>
__global__ void __launch_bounds__(256) probe_unit_kernel(const ProbeArgs a) {
    constexpr int UR = 2, UC = 2, THREADS = 256;
    constexpr int N = 128 / static_cast<int>(sizeof(T));
    constexpr int VPE = 16 / static_cast<int>(sizeof(T));
    constexpr int P = (VARIANT == SWZ_T_PADDED) ? N + 1 : N;
    constexpr int TR = UR * N, TC = UC * N;
    constexpr int ITER = TR * TC / VPE / THREADS;
    __shared__ T sm[UR * UC * N * P];
    const int tid = threadIdx.x;
    auto phys = [](int ir, int ic) -> int { return VARIANT == SWZ_T_SWIZZLED ? (ic ^ ir) : ic; };
    uint32_t acc = tid;
    for (int it = 0; it < a.iters; ++it) {
        uint4 v[ITER];
#pragma unroll
        for (int k = 0; k < ITER; ++k) {
            v[k] = make_uint4(acc + k, acc ^ it, acc + it, acc ^ k);
            if (a.gsrc) {
                const uint4 gv = ld_stream16(a.gsrc + probe_gvec(a, it, k, ITER));
                v[k].x ^= gv.x; v[k].y ^= gv.y; v[k].z ^= gv.z; v[k].w ^= gv.w;
            }
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
            acc ^= fold(o);
            if (a.gdst) st_stream16(a.gdst + probe_gvec(a, it, k, ITER), o);
        }
        __syncthreads();
    }
    if (a.sink && tid == 0) a.sink[blockIdx.x] = acc;
}

// --------------------------------------------------------------- 2 bytes --
// The 64 x 64 staging of the 16-bit transpose: 128 threads, 16-byte fill
// stores, ldmatrix .x4 .trans drain.
template <int VARIANT>
__global__ void __launch_bounds__(128) probe_16_kernel(const ProbeArgs a) {
    constexpr int THREADS = 128;
    constexpr int PITCH = (VARIANT == SWZ_T_PADDED) ? 72 : 64;
    constexpr bool OUT_TILE = VARIANT == SWZ_T_TMA;
    __shared__ __align__(1024) uint16_t sm[64 * PITCH];
    __shared__ __align__(1024) uint16_t out_sm[OUT_TILE ? 64 * 64 : 8];
    const int tid = threadIdx.x;
    auto chunk = [](int row, int ch) -> int {
        return (VARIANT == SWZ_T_SWIZZLED || VARIANT == SWZ_T_TMA) ? (ch ^ (row & 7)) : ch;
    };
    uint32_t acc = tid;
    for (int it = 0; it < a.iters; ++it) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[k] = make_uint4(acc + k, acc ^ it, acc + it, acc ^ k);
            if (a.gsrc) {
                const uint4 gv = ld_stream16(a.gsrc + probe_gvec(a, it, k, 4));
                v[k].x ^= gv.x; v[k].y ^= gv.y; v[k].z ^= gv.z; v[k].w ^= gv.w;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int id = k * THREADS + tid, ch = id & 7, row = id >> 3;
            *reinterpret_cast<uint4 *>(sm + row * PITCH + chunk(row, ch) * 8) = v[k];
        }
        __syncthreads();
        const int lane = tid & 31, warp = tid >> 5;
        const int m = lane >> 3, i = lane & 7;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int xi = warp * 4 + k;
            const int cb = xi & 7, rbg = (xi >> 3) * 4;
            const int row = (rbg + m) * 8 + i;
            uint32_t a0, a1, a2, a3;
            probe_ldmatrix_x4_trans(smem_u32(sm + row * PITCH + chunk(row, cb) * 8), a0, a1, a2, a3);
            if constexpr (OUT_TILE) {
                // block (rbg + m, cb) transposed goes to output block (cb, rbg + m)
                const int orow = cb * 8 + i;
                asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(
                                 smem_u32(out_sm + orow * 64 + (((rbg + m) ^ (orow & 7)) << 3))),
                             "r"(a0), "r"(a1), "r"(a2), "r"(a3)
                             : "memory");
            }
            const uint4 o = make_uint4(a0, a1, a2, a3);
            acc ^= fold(o);
            if (a.gdst) st_stream16(a.gdst + probe_gvec(a, it, k, 4), o);
        }
        __syncthreads();
    }
    if (a.sink && tid == 0) a.sink[blockIdx.x] = acc;
}

// ---------------------------------------------------------------- 1 byte --
// The 128 x 128 byte staging of the 1-byte transpose: 256 threads, 16-byte
// fill stores, 4-byte drain loads from 16 consecutive rows.
__global__ void __launch_bounds__(256) probe_8_kernel(const ProbeArgs a) {
    constexpr int T = 128, THREADS = 256;
    __shared__ __align__(16) uint8_t sm[T * T];
    const int tid = threadIdx.x;
    auto at = [](int row, int col) -> int { return row * T + ((((col >> 4) ^ (row >> 4)) & 7) << 4) + (col & 15); };
    uint32_t acc = tid;
    for (int it = 0; it < a.iters; ++it) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[k] = make_uint4(acc + k, acc ^ it, acc + it, acc ^ k);
            if (a.gsrc) {
                const uint4 gv = ld_stream16(a.gsrc + probe_gvec(a, it, k, 4));
                v[k].x ^= gv.x; v[k].y ^= gv.y; v[k].z ^= gv.z; v[k].w ^= gv.w;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int id = k * THREADS + tid, row = id >> 3, ch = id & 7;
            *reinterpret_cast<uint4 *>(sm + at(row, ch * 16)) = v[k];
        }
        __syncthreads();
        const int lane = tid & 31, warp = tid >> 5;
        const int g = lane & 7, q = 4 * warp + (lane >> 3);
#pragma unroll
        for (int aa = 0; aa < 4; ++aa) {
            uint4 o;
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = *reinterpret_cast<const uint32_t *>(sm + at(16 * g + 4 * aa + k, 4 * q));
            o = make_uint4(w[0], w[1], w[2], w[3]);
            acc ^= fold(o);
            if (a.gdst) st_stream16(a.gdst + probe_gvec(a, it, aa, 4), o);
        }
        __syncthreads();
    }
    if (a.sink && tid == 0) a.sink[blockIdx.x] = acc;
}

}  // namespace
}  // namespace swz

extern "C" swz_status swz_staging_probe(int esize, int variant, int iters, const void *gsrc, void *gdst,
                                        int64_t gbytes, uint32_t *sink, int64_t ctas, void *stream) {
    using namespace swz;
    if (iters < 0 || ctas < 0 || ctas > 0x7fffffffLL) return SWZ_ERR_SHAPE;
    if (variant != SWZ_T_SWIZZLED && variant != SWZ_T_UNSWIZZLED && variant != SWZ_T_PADDED &&
        !(variant == SWZ_T_TMA && esize == 2))
        return SWZ_ERR_PARAM;
    if (esize != 1 && esize != 2 && esize != 4 && esize != 8) return SWZ_ERR_PARAM;
    if (esize == 1 && variant != SWZ_T_SWIZZLED) return SWZ_ERR_PARAM;
    if ((gsrc || gdst) && (gbytes < 16 || gbytes % 16 != 0)) return SWZ_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(gsrc) | reinterpret_cast<uintptr_t>(gdst)) & 15u) return SWZ_ERR_ALIGN;
    if (gsrc && gdst && ranges_overlap(gsrc, gbytes, gdst, gbytes)) return SWZ_ERR_ALIAS;
    if (iters == 0 || ctas == 0) return SWZ_OK;
    ProbeArgs a;
    a.gsrc = static_cast<const uint4 *>(gsrc);
    a.gdst = static_cast<uint4 *>(gdst);
    a.gvecs = gbytes / 16;
    a.iters = iters;
    a.sink = sink;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 g(static_cast<unsigned>(ctas));
    switch (esize) {
        case 1: probe_8_kernel<<<g, 256, 0, st>>>(a); break;
        case 2:
            if (variant == SWZ_T_SWIZZLED) probe_16_kernel<SWZ_T_SWIZZLED><<<g, 128, 0, st>>>(a);
            else if (variant == SWZ_T_UNSWIZZLED) probe_16_kernel<SWZ_T_UNSWIZZLED><<<g, 128, 0, st>>>(a);
            else if (variant == SWZ_T_TMA) probe_16_kernel<SWZ_T_TMA><<<g, 128, 0, st>>>(a);
            else probe_16_kernel<SWZ_T_PADDED><<<g, 128, 0, st>>>(a);
            break;
        case 4:
            if (variant == SWZ_T_SWIZZLED) probe_unit_kernel<uint32_t, SWZ_T_SWIZZLED><<<g, 256, 0, st>>>(a);
            else if (variant == SWZ_T_UNSWIZZLED) probe_unit_kernel<uint32_t, SWZ_T_UNSWIZZLED><<<g, 256, 0, st>>>(a);
            else probe_unit_kernel<uint32_t, SWZ_T_PADDED><<<g, 256, 0, st>>>(a);
            break;
        default:
            if (variant == SWZ_T_SWIZZLED) probe_unit_kernel<unsigned long long, SWZ_T_SWIZZLED><<<g, 256, 0, st>>>(a);
            else if (variant == SWZ_T_UNSWIZZLED) probe_unit_kernel<unsigned long long, SWZ_T_UNSWIZZLED><<<g, 256, 0, st>>>(a);
            else probe_unit_kernel<unsigned long long, SWZ_T_PADDED><<<g, 256, 0, st>>>(a);
            break;
    }
    return launch_status();
}
