// swz_tma.cu -- 16-bit transpose whose tiles enter shared memory through TMA
// tensor copies with the hardware 128-byte swizzle (sm_103a).
//
// The hardware 128-byte swizzle mode places 16-byte chunk c of box row r at
// chunk position c ^ (r mod 8) inside each 1024-byte span, which is the
// byte-address Swizzle<3,4,3> ("CuTe Swizzle 学习手册", sections "Sw<3,4,3>
// vs Sw<3,3,3>" and "H100 TMA + Swizzle"): with 64-element (128-byte) box
// rows it is exactly the layout of the SWZ_T_SWIZZLED 16-bit kernel, so the
// same conflict-free transposing matrix loads drain it.
//
// One 64 x 64 tile per CTA (a grid of one CTA per tile, up to 12 resident per
// SM): one thread issues the tile's tensor load, every thread waits on the
// tile's mbarrier, and the drain reads 8 x 8 blocks with ldmatrix .trans.
// When the output rows are whole 16-byte vectors (TSTORE) the blocks go out
// through stmatrix into an output tile under the same 128-byte swizzle and
// one tensor store; otherwise element by element from the shared tile.
// The hardware block scheduler hands out tiles in order, so the tiles in
// flight stay a compact band of the matrix; a persistent grid that walked
// tiles blockIdx.x, +gridDim.x, ... with a ring of stages drifted apart and
// ran 5-10% slower on the 16384^2 matrix.
//
// Every wait on the mbarrier is bounded by a time limit; on expiry the kernel
// records SWZ_ERR_TIMEOUT in a status word, waits (again bounded) for its own
// copy still in flight, and returns; swz_device_status() reports it.
#include "swz_tma_common.cuh"

#include <climits>
#include <mutex>

namespace swz {
namespace {

constexpr int kTile = 64;                        // 64 x 64 elements
constexpr int kTileBytes = kTile * kTile * 2;    // 8 KiB
constexpr int kThreads = 128;

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &d0, uint32_t &d1,
                                                  uint32_t &d2, uint32_t &d3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(addr));
}

__device__ __forceinline__ void stmatrix_x4(uint32_t addr, uint32_t d0, uint32_t d1, uint32_t d2, uint32_t d3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(d0), "r"(d1),
                 "r"(d2), "r"(d3)
                 : "memory");
}

struct TmaArgs {
    uint16_t *dst;
    int64_t R, C, tiles_c, n_tiles;
    int issue_copies;   // 0 only in the timeout self-tests: no copy is issued, every wait expires
    uint64_t wait_ns;
    uint32_t *status;   // status word that an expired wait reports to
};

// Dynamic shared memory of the kernel: the input tile, the output tile when
// TSTORE, and up to 1 KiB of slack to align them to the swizzle's 1024 bytes.
constexpr int tma_smem_bytes(bool tstore) { return (tstore ? 2 : 1) * kTileBytes + 1024; }

template <bool TSTORE>
__global__ void __launch_bounds__(kThreads)
    transpose16_tma_kernel(const __grid_constant__ CUtensorMap map_in, const __grid_constant__ CUtensorMap map_out,
                           const TmaArgs a) {
    pdl_launch_dependents();
    pdl_wait();  // before the first tensor copy
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t ib = (raw + 1023u) & ~1023u;  // the 128-byte swizzle repeats every 1024 bytes
    const uint32_t ob = ib + kTileBytes;
    const uint16_t *sm = reinterpret_cast<const uint16_t *>(smem_raw + (ib - raw));
    const int tid = threadIdx.x;
    const uint32_t b = smem_u32(&bar);

    if (tid == 0) {
        mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    const int lane = tid & 31, warp = tid >> 5;
    const int m = lane >> 3, i8 = lane & 7;  // matrix addressed by this lane, its row
    uint32_t it = 0;                         // tiles done by this CTA (the barrier's phase)
    for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x, ++it) {
        const int64_t tr = t / a.tiles_c, tc = t - tr * a.tiles_c;
        if (tid == 0 && a.issue_copies) {
            mbar_expect_tx(b, kTileBytes);
            tma_load_2d(ib, &map_in, static_cast<int>(tc * kTile), static_cast<int>(tr * kTile), b);
        }
        const bool ok = mbar_wait_bounded(b, it & 1u, a.wait_ns);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(a.status, 1u << SWZ_ERR_TIMEOUT);
                // let this CTA's copy still in flight land before the CTA exits
                if (a.issue_copies) mbar_wait_bounded(b, it & 1u, a.wait_ns);
                if (TSTORE) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            }
            return;
        }
        if constexpr (TSTORE) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int xi = warp * 4 + k;
                const int cb = xi & 7, rbg = (xi >> 3) * 4;
                const int row = (rbg + m) * 8 + i8;   // input tile row this lane addresses
                uint32_t d0, d1, d2, d3;
                ldmatrix_x4_trans(ib + row * 128 + ((cb ^ (row & 7)) << 4), d0, d1, d2, d3);
                // block (rbg + m, cb) transposed lands at output block (cb, rbg + m)
                const int orow = cb * 8 + i8;
                stmatrix_x4(ob + orow * 128 + (((rbg + m) ^ (orow & 7)) << 4), d0, d1, d2, d3);
            }
            // the shared writes are ordered before the tensor store that reads them,
            // and the shared reads before the next tensor load into the input tile
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();
            if (tid == 0) {
                tma_store_2d(&map_out, static_cast<int>(tr * kTile), static_cast<int>(tc * kTile), ob);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                // the output tile is read before this CTA rewrites it or exits
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            }
        } else {
            const int64_t r0 = tr * kTile, c0 = tc * kTile;
            for (int idx = tid; idx < kTile * kTile; idx += kThreads) {
                const int ocl = idx / kTile, orow = idx % kTile;
                if (c0 + ocl < a.C && r0 + orow < a.R)
                    a.dst[(c0 + ocl) * a.R + r0 + orow] = sm[orow * 64 + (((ocl >> 3) ^ (orow & 7)) << 3) + (ocl & 7)];
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncthreads();  // the tiles are free for the next tile of this CTA
    }
}

// ---- host side ---------------------------------------------------------

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
uint32_t *g_status[kMaxDevices] = {};

}  // namespace

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// The per-device status word (allocated once per device, on first use).
uint32_t *device_status_word(bool create) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status[dev] && create) {
        uint32_t *p = nullptr;
        if (cudaMalloc(&p, sizeof(uint32_t)) != cudaSuccess) return nullptr;
        if (cudaMemset(p, 0, sizeof(uint32_t)) != cudaSuccess) { cudaFree(p); return nullptr; }
        g_status[dev] = p;
    }
    return g_status[dev];
}

swz_status transpose_launch(void *dst, const void *src, int64_t R, int64_t C, int esize, int variant,
                            cudaStream_t st);

// Encodes the tensor maps and launches transpose16_tma_kernel: the output
// leaves by tensor store when its rows are whole 16-byte vectors (dst 16-byte
// aligned, rows a multiple of 8), element by element otherwise.  Expired waits
// report to `status`.  The caller has checked that TMA applies (src 16-byte
// aligned, cols a multiple of 8, rows and cols below 2^31).
swz_status tma_transpose_enqueue(EncodeTiledFn encode, void *dst, const void *src, int64_t R, int64_t C,
                                 cudaStream_t st, int issue_copies, uint64_t wait_ns, uint32_t *status) {
    CUtensorMap map_in, map_out;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(R)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(C) * 2};
    const cuuint32_t box[2] = {kTile, kTile};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&map_in, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(src), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SWZ_ERR_CUDA;
    const bool tstore = ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) && (R % 8 == 0);
    if (tstore) {
        // the output (C x R, rows of R elements) goes out through its own tensor map
        const cuuint64_t odim[2] = {static_cast<cuuint64_t>(R), static_cast<cuuint64_t>(C)};
        const cuuint64_t ostride[1] = {static_cast<cuuint64_t>(R) * 2};
        if (encode(&map_out, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, dst, odim, ostride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SWZ_ERR_CUDA;
    } else {
        map_out = map_in;  // not read by the element-wise drain
    }
    TmaArgs a;
    a.dst = static_cast<uint16_t *>(dst);
    a.R = R;
    a.C = C;
    a.tiles_c = (C + kTile - 1) / kTile;
    a.n_tiles = ((R + kTile - 1) / kTile) * a.tiles_c;
    a.issue_copies = issue_copies;
    a.wait_ns = wait_ns;
    a.status = status;
    // one CTA per tile; past the grid limit each CTA takes every gridDim.x-th tile
    const unsigned grid = static_cast<unsigned>(a.n_tiles < INT_MAX ? a.n_tiles : INT_MAX);
    if (tstore)
        return launched(launch_pdl(transpose16_tma_kernel<true>, dim3(grid), dim3(kThreads), tma_smem_bytes(true),
                                   st, map_in, map_out, a));
    return launched(launch_pdl(transpose16_tma_kernel<false>, dim3(grid), dim3(kThreads), tma_smem_bytes(false), st,
                               map_in, map_out, a));
}

swz_status transpose_tma_run(void *dst, const void *src, int64_t R, int64_t C, cudaStream_t st,
                             int issue_copies, uint64_t wait_ns) {
    // TMA needs 16-byte aligned source rows and int32 coordinates; otherwise
    // the shared-memory-staged swizzled kernel does the same job.
    const bool tma_ok = (reinterpret_cast<uintptr_t>(src) & 15u) == 0 && (C % 8) == 0 && R < (1LL << 31) &&
                        C < (1LL << 31);
    EncodeTiledFn encode = encode_fn();
    if (!tma_ok || !encode) return transpose_launch(dst, src, R, C, 2, SWZ_T_SWIZZLED, st);
    uint32_t *status = device_status_word(true);
    if (!status) return SWZ_ERR_CUDA;
    return tma_transpose_enqueue(encode, dst, src, R, C, st, issue_copies, wait_ns, status);
}

swz_status transpose_tma_launch(void *dst, const void *src, int64_t R, int64_t C, cudaStream_t st) {
    return transpose_tma_run(dst, src, R, C, st, 1, kWaitLimitNs);
}

}  // namespace swz

extern "C" {

// Waits for `stream`, then reads and clears the calling device's status word.
swz_status swz_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SWZ_ERR_CUDA;
    uint32_t *w = swz::device_status_word(false);
    if (!w) return SWZ_OK;
    uint32_t v = 0;
    if (cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return SWZ_ERR_CUDA;
    if (v && cudaMemset(w, 0, sizeof v) != cudaSuccess) return SWZ_ERR_CUDA;
    return (v & (1u << SWZ_ERR_TIMEOUT)) ? SWZ_ERR_TIMEOUT : SWZ_OK;
}

// Self-test of the bounded wait: runs the TMA transpose kernel with no copy
// issued, so every mbarrier wait expires after wait_ns nanoseconds and the
// kernel must record SWZ_ERR_TIMEOUT and return.  dst is not written.
swz_status swz_selftest_tma_timeout(void *dst, const void *src, int64_t rows, int64_t cols,
                                    uint64_t wait_ns, void *stream) {
    if (!dst || !src) return SWZ_ERR_NULL;
    if (rows <= 0 || cols <= 0 || cols % 8 != 0) return SWZ_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) != 0) return SWZ_ERR_ALIGN;
    return swz::transpose_tma_run(dst, src, rows, cols, static_cast<cudaStream_t>(stream), 0, wait_ns);
}

}  // extern "C"

// ---- allocation-free variant of the TMA transpose ------------------------
//
// For callers that must not have the library allocate device memory: the
// SWZ_T_TMA path above makes one cudaMalloc (its status word) on the first
// call on each device.  This variant runs the same kernel with its status
// word taken from a fixed array in the library's own device data instead.
namespace swz {
namespace {

// The scratch of the allocation-free call: word 0 is the status word the
// kernel sets when a bounded wait gives up.  256 bytes at file scope; every
// GPU that loads the library holds one copy until the process exits.
constexpr int kNoAllocScratchWords = 64;
constexpr int kNoAllocWordsNeeded = 1;  // one status word, whatever the matrix size
static_assert(kNoAllocWordsNeeded <= kNoAllocScratchWords, "scratch array too small");
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchWords];

std::mutex g_noalloc_mu;
uint32_t *g_noalloc_addr[kMaxDevices] = {};

// Set-up, once per device, with that device current: the device address of
// g_noalloc_scratch.  (In host code the array's name only stands for the
// symbol; a kernel must be given this address.)
uint32_t *noalloc_scratch(int dev) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_noalloc_addr[dev] = static_cast<uint32_t *>(p);
    }
    return g_noalloc_addr[dev];
}

}  // namespace
}  // namespace swz

namespace swz {
namespace {

// The allocation-free call; issue_copies = 0 and a short wait_ns only in its
// timeout self-test (no copy is issued, so every bounded wait expires).
swz_status noalloc_run(void *dst, const void *src, int64_t rows, int64_t cols, uint32_t *timed_out,
                       cudaStream_t st, int issue_copies, uint64_t wait_ns) {
    if (timed_out) *timed_out = 0;
    if (rows < 0 || cols < 0) return SWZ_ERR_SHAPE;
    // the largest request: TMA coordinates are 32-bit
    if (rows >= (1LL << 31) || cols >= (1LL << 31)) return SWZ_ERR_SHAPE;
    if (rows == 0 || cols == 0) return SWZ_OK;
    // rows * cols * 2 stays below 2^63 for rows, cols < 2^31; checked all the same
    if (rows > INT64_MAX / 2 / cols) return SWZ_ERR_SHAPE;
    if (!dst || !src) return SWZ_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 1u) return SWZ_ERR_ALIGN;
    const int64_t n_bytes = rows * cols * 2;
    if (ranges_overlap(dst, n_bytes, src, n_bytes)) return SWZ_ERR_ALIAS;

    EncodeTiledFn encode = encode_fn();
    const bool tma_ok = encode && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 && (cols % 8) == 0;
    if (!tma_ok) {
        if (!issue_copies) return encode ? SWZ_ERR_SHAPE : SWZ_ERR_CUDA;  // the self-test needs the TMA kernel
        // same fallback as SWZ_T_TMA: the shared-memory-staged swizzled kernel, no scratch
        const swz_status s = transpose_launch(dst, src, rows, cols, 2, SWZ_T_SWIZZLED, st);
        if (s == SWZ_OK && timed_out && cudaStreamSynchronize(st) != cudaSuccess) return SWZ_ERR_CUDA;
        return s;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SWZ_ERR_CUDA;
    uint32_t *scratch = noalloc_scratch(dev);
    if (!scratch) return SWZ_ERR_CUDA;
    // the array keeps the previous call's contents: the status word must start at zero
    if (cudaMemsetAsync(scratch, 0, kNoAllocWordsNeeded * sizeof(uint32_t), st) != cudaSuccess)
        return SWZ_ERR_CUDA;

    const swz_status s = tma_transpose_enqueue(encode, dst, src, rows, cols, st, issue_copies, wait_ns, scratch);
    if (s != SWZ_OK || !timed_out) return s;
    uint32_t v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess ||
        cudaMemcpy(&v, scratch, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SWZ_ERR_CUDA;
    if (v & (1u << SWZ_ERR_TIMEOUT)) {
        *timed_out = 1;
        return SWZ_ERR_TIMEOUT;
    }
    return SWZ_OK;
}

}  // namespace
}  // namespace swz

extern "C" swz_status swz_transpose_tma_noalloc(void *dst, const void *src, int64_t rows, int64_t cols,
                                                uint32_t *timed_out, void *stream) {
    return swz::noalloc_run(dst, src, rows, cols, timed_out, static_cast<cudaStream_t>(stream), 1,
                            swz::kWaitLimitNs);
}

// Self-test of the allocation-free call's timeout report: the same call with
// no tensor copy issued, so every bounded wait gives up after wait_ns and the
// kernel records the expiry in the fixed array's status word.
extern "C" swz_status swz_selftest_noalloc_timeout(void *dst, const void *src, int64_t rows, int64_t cols,
                                                   uint64_t wait_ns, uint32_t *timed_out, void *stream) {
    if (!timed_out) return SWZ_ERR_NULL;
    if (!dst || !src) return SWZ_ERR_NULL;
    if (rows <= 0 || cols <= 0 || cols % 8 != 0) return SWZ_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) != 0) return SWZ_ERR_ALIGN;
    return swz::noalloc_run(dst, src, rows, cols, timed_out, static_cast<cudaStream_t>(stream), 0, wait_ns);
}
