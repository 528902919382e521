// swz_tma_relayout.cu -- relayout through the tensor-memory accelerator's
// hardware swizzle (sm_103a).
//
// A TMA tensor copy in the 32-, 64- or 128-byte swizzle mode XORs bits
// [4, 4 + B) of the shared-memory byte address with bits [7, 7 + B), B = 1, 2,
// 3: the byte-address Swizzle<B,4,3>, i.e. element Swizzle<B, 4 - log2 e, 3> on
// e-byte elements ("CuTe Swizzle 学习手册", sections "Sw<3,4,3> vs Sw<3,3,3>"
// and "H100 TMA + Swizzle").  The 128-byte mode with 32-byte atoms XORs bits
// [5, 7) with bits [7, 9): the byte-address Swizzle<2,5,2>.  The buffer is
// viewed as rows of the swizzle span (32, 64 or 128 bytes) and moved in 8 KiB
// chunks, one per CTA: a swizzled tensor load puts
// the logical byte at offset i of a chunk at shared offset sw(i), then every
// thread copies its 16-byte vectors out to dst in order, so dst[sw(i)] =
// src[i].  Every hardware mode is its own inverse (the field it reads sits
// at or above the field it writes plus its width), so the inverse relayout
// dst[i] = src[sw(i)] is the same copy.  (An inverse that filled shared
// memory with 16-byte stores and left by a swizzled tensor store ran at 6.73
// against 6.9 TB/s, and its shared stores collided with the tensor store's
// shared reads on 11% of their wavefronts.)
// Each chunk covers whole swizzle periods (at most 1 KiB) of whole tiles, so
// the tile-local swizzle equals the swizzle of the chunk-local offset.  The
// kernel waits on its loads with bounded mbarrier waits (kWaitLimitNs) and
// records an expiry in the per-device status word.
#include "swz_tma_common.cuh"

#include <climits>

namespace swz {

swz_status relayout_launch(void *dst, const void *src, int64_t n_tiles, int64_t tile_elems, int esize, int B,
                           int M, int S, int direction, cudaStream_t st);

namespace {

constexpr int kChunk = 8192;                         // bytes per tensor copy
constexpr int kThreads = 256;
constexpr int kVecs = kChunk / 16 / kThreads;        // 16-byte vectors per thread per chunk
// One chunk per CTA: a grid of one CTA per chunk (8 resident per SM) keeps the
// chunks in flight a compact band of the buffer.  A persistent grid of 2 CTAs
// per SM with 3 chunks in flight each ran at 6.84 against 7.06 TB/s (1 GiB,
// 128-byte mode); past the grid limit a CTA takes every gridDim.x-th chunk and
// loads the next while it stores the current one.
constexpr int kRing = 1;

struct TmaRelayoutArgs {
    uint8_t *dst;
    const uint8_t *src;
    int64_t bytes;          // the whole buffer
    int64_t n_chunks;
    int rows_per_chunk;     // kChunk / swizzle span
    uint64_t wait_ns;
    uint32_t *status;
};

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// 16-byte vectors of chunk c that hold data (the last chunk may be short)
__device__ __forceinline__ int chunk_vecs(const TmaRelayoutArgs &a, int64_t c) {
    const int64_t left = a.bytes - c * kChunk;
    return static_cast<int>((left < kChunk ? left : kChunk) / 16);
}

__global__ void __launch_bounds__(kThreads)
    relayout_tma_kernel(const __grid_constant__ CUtensorMap map, const TmaRelayoutArgs a) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[kRing];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;  // the swizzle is computed from address bits
    const uint32_t bar0 = smem_u32(&bars[0]);
    const int tid = threadIdx.x;
    // a tensor box always transfers its full size (rows past the end are zero-filled)
    auto issue = [&](int s, int64_t c) {
        mbar_expect_tx(bar0 + 8u * s, kChunk);
        tma_load_2d(base + s * kChunk, &map, 0, static_cast<int>(c * a.rows_per_chunk), bar0 + 8u * s);
    };
    if (tid == 0) {
        for (int s = 0; s < kRing; ++s) mbar_init(bar0 + 8u * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        for (int s = 0; s < kRing; ++s) {
            const int64_t c = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (c < a.n_chunks) issue(s, c);
        }
    }
    __syncthreads();
    for (int64_t it = 0;; ++it) {
        const int64_t c = blockIdx.x + it * gridDim.x;
        if (c >= a.n_chunks) break;
        const int s = static_cast<int>(it % kRing);
        const bool ok = mbar_wait_bounded(bar0 + 8u * s, static_cast<uint32_t>((it / kRing) & 1), a.wait_ns);
        if (!__syncthreads_and(ok)) {
            if (tid == 0) {
                atomicOr(a.status, 1u << SWZ_ERR_TIMEOUT);
                // let the loads still in flight (iterations it .. it + kRing - 1) land
                for (int64_t j = it; j < it + kRing; ++j) {
                    if (blockIdx.x + j * gridDim.x >= a.n_chunks) break;
                    mbar_wait_bounded(bar0 + 8u * static_cast<uint32_t>(j % kRing),
                                      static_cast<uint32_t>((j / kRing) & 1), a.wait_ns);
                }
            }
            return;
        }
        const int nv = chunk_vecs(a, c);
        uint4 v[kVecs];
#pragma unroll
        for (int k = 0; k < kVecs; ++k) {
            const int idx = k * kThreads + tid;
            if (idx < nv) v[k] = lds16(base + s * kChunk + idx * 16);
        }
        // every thread orders its reads of buffer s before the tensor copy
        // that refills it (the copy writes through the async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            const int64_t cn = c + static_cast<int64_t>(kRing) * gridDim.x;
            if (cn < a.n_chunks) issue(s, cn);
        }
#pragma unroll
        for (int k = 0; k < kVecs; ++k) {
            const int idx = k * kThreads + tid;
            if (idx < nv) st_stream16(a.dst + c * kChunk + idx * 16, v[k]);
        }
    }
}

// The hardware swizzle modes as byte-address Swizzle<B, Mb, S> (measured on
// GB300 with tensor loads of every element size): 16-byte chunks within 32-,
// 64- and 128-byte spans XOR-ed with the row (bits 7..), and 32-byte chunks
// within a 128-byte span XOR-ed with the row mod 4.
struct HwMode {
    int B, Mb, S;
    int span;  // bytes per tensor row: the swizzle span
    CUtensorMapSwizzle mode;
};
constexpr int kHwModes = 4;
const HwMode kModes[kHwModes] = {
    {1, 4, 3, 32, CU_TENSOR_MAP_SWIZZLE_32B},
    {2, 4, 3, 64, CU_TENSOR_MAP_SWIZZLE_64B},
    {3, 4, 3, 128, CU_TENSOR_MAP_SWIZZLE_128B},
    {2, 5, 2, 128, CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B},
};

// Index into kModes of the hardware mode that runs this request, or -1 when
// the register kernels run it.
int tma_plan(const void *dst, const void *src, int64_t bytes, int64_t tile_bytes, int esize, int B, int M, int S) {
    int k = 0;
    while ((1 << k) < esize) ++k;
    const bool aligned = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
    if (!aligned || !encode_fn()) return -1;
    for (int i = 0; i < kHwModes; ++i) {
        const HwMode &h = kModes[i];
        if (B != h.B || S != h.S || M + k != h.Mb) continue;
        const int64_t period = int64_t(1) << (h.B + h.Mb + h.S);  // bytes
        if (tile_bytes % period != 0 || bytes / h.span >= (int64_t(1) << 31)) return -1;
        return i;
    }
    return -1;
}

}  // namespace

// Which path swz_relayout_tma takes (arguments validated by the caller):
// 0 for the register kernels, else 1 + the index of the hardware mode.
int relayout_tma_path(const void *dst, const void *src, int64_t n_tiles, int64_t tile_elems, int esize, int B,
                      int M, int S) {
    return 1 + tma_plan(dst, src, n_tiles * tile_elems * esize, tile_elems * esize, esize, B, M, S);
}

// Arguments are validated by the caller (swz_relayout_tma in swz_abi.cu).
swz_status relayout_tma_launch(void *dst, const void *src, int64_t n_tiles, int64_t tile_elems, int esize, int B,
                               int M, int S, int direction, cudaStream_t st) {
    const int64_t tile_bytes = tile_elems * esize;
    const int64_t bytes = n_tiles * tile_bytes;
    const int plan = tma_plan(dst, src, bytes, tile_bytes, esize, B, M, S);
    if (plan < 0) return relayout_launch(dst, src, n_tiles, tile_elems, esize, B, M, S, direction, st);
    const HwMode &h = kModes[plan];
    EncodeTiledFn encode = encode_fn();
    uint32_t *status = device_status_word(true);
    if (!status) return SWZ_ERR_CUDA;

    const int64_t span = h.span;
    CUtensorMap map;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(span), static_cast<cuuint64_t>(bytes / span)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(span)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(span), static_cast<cuuint32_t>(kChunk / span)};
    const cuuint32_t estride[2] = {1, 1};
    (void)direction;  // every hardware mode is its own inverse: both directions are the same copy
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(src), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, h.mode, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SWZ_ERR_CUDA;

    TmaRelayoutArgs a;
    a.dst = static_cast<uint8_t *>(dst);
    a.src = static_cast<const uint8_t *>(src);
    a.bytes = bytes;
    a.n_chunks = (bytes + kChunk - 1) / kChunk;
    a.rows_per_chunk = static_cast<int>(kChunk / span);
    a.wait_ns = kWaitLimitNs;
    a.status = status;
    const int64_t grid = a.n_chunks < INT_MAX ? a.n_chunks : INT_MAX;
    const dim3 g(static_cast<unsigned>(grid));
    return launched(launch_pdl(relayout_tma_kernel, g, dim3(kThreads), kRing * kChunk + 1024, st, map, a));
}

}  // namespace swz
