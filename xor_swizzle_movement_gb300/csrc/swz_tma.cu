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
// When the output rows are whole 16-byte vectors the output leaves by TMA
// too (transpose16_tma_ls_kernel): ldmatrix .trans, then stmatrix into an
// output tile under the same 128-byte swizzle, then one tensor store per tile.
// Otherwise the drained rows leave by 16-byte stores (transpose16_tma_kernel).
//
// Persistent kernels: each CTA walks tiles blockIdx.x, +gridDim.x, ...; a
// ring of kStages shared buffers keeps kStages tile loads in flight while the
// current tile is drained.  One elected thread issues the copies; each buffer
// has an mbarrier that the copy completes.  Every wait on an mbarrier is
// bounded by a time limit; on expiry the kernel records SWZ_ERR_TIMEOUT in a
// per-device status word, waits (again bounded) for its own copies still in
// flight, and returns; swz_device_status() reports it to the host.
#include "swz_tma_common.cuh"

#include <mutex>

namespace swz {
namespace {

constexpr int kStages = 4;
constexpr int kTile = 64;                        // 64 x 64 elements
constexpr int kTileBytes = kTile * kTile * 2;    // 8 KiB
constexpr int kThreads = 128;

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &d0, uint32_t &d1,
                                                  uint32_t &d2, uint32_t &d3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t pick4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, int i) {
    const uint32_t lo = (i & 1) ? a1 : a0;
    const uint32_t hi = (i & 1) ? a3 : a2;
    return (i & 2) ? hi : lo;
}

struct TmaArgs {
    uint16_t *dst;
    int64_t R, C, tiles_c, n_tiles;
    int vec_store_ok;
    int issue_copies;   // 0 only in the timeout self-test: no copy is issued, every wait expires
    uint64_t wait_ns;
    uint32_t *status;   // per-device status word
};

__global__ void __launch_bounds__(kThreads)
    transpose16_tma_kernel(const __grid_constant__ CUtensorMap map, const TmaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[kStages];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // the 128-byte swizzle repeats every 1024 bytes
    uint8_t *const gbase = smem_raw + (base - raw);
    const int tid = threadIdx.x;
    const uint32_t bar0 = smem_u32(&bars[0]);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8u * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    auto issue = [&](int s, int64_t t) {
        const int64_t tr = t / a.tiles_c, tc = t - tr * a.tiles_c;
        mbar_expect_tx(bar0 + 8u * s, kTileBytes);
        tma_load_2d(base + s * kTileBytes, &map, static_cast<int>(tc * kTile), static_cast<int>(tr * kTile),
                    bar0 + 8u * s);
    };
    if (tid == 0 && a.issue_copies) {
        for (int s = 0; s < kStages; ++s) {
            const int64_t t = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (t < a.n_tiles) issue(s, t);
        }
    }

    const int lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, kk = lane & 3, m = lane >> 3, i8 = lane & 7;
    int64_t it = 0;
    for (;; ++it) {
        const int64_t t = blockIdx.x + it * gridDim.x;
        if (t >= a.n_tiles) break;
        const int s = static_cast<int>(it % kStages);
        const uint32_t parity = static_cast<uint32_t>((it / kStages) & 1);
        const bool ok = mbar_wait_bounded(bar0 + 8u * s, parity, a.wait_ns);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicOr(a.status, 1u << SWZ_ERR_TIMEOUT);
            // let this CTA's copies still in flight land before the CTA exits
            if (a.issue_copies) {
                for (int64_t j = it; j < it + kStages; ++j) {
                    const int64_t tj = blockIdx.x + j * gridDim.x;
                    if (tj >= a.n_tiles) break;
                    mbar_wait_bounded(bar0 + 8u * static_cast<uint32_t>(j % kStages),
                                      static_cast<uint32_t>((j / kStages) & 1), a.wait_ns);
                }
            }
            return;
        }
        const uint16_t *sm = reinterpret_cast<const uint16_t *>(gbase + s * kTileBytes);
        const int64_t tr = t / a.tiles_c, tc = t - tr * a.tiles_c;
        const int64_t r0 = tr * kTile, c0 = tc * kTile;
        if (a.vec_store_ok && r0 + kTile <= a.R && c0 + kTile <= a.C) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int xi = warp * 4 + k;
                const int cb = xi & 7, rbg = (xi >> 3) * 4;
                const int row = (rbg + m) * 8 + i8;
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4_trans(base + s * kTileBytes + row * 128 + ((cb ^ (row & 7)) << 4), a0, a1, a2, a3);
                uint32_t b0 = 0, b1 = 0, b2 = 0, b3 = 0;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int from = kk ^ r;
                    const uint32_t send = pick4(a0, a1, a2, a3, from);
                    const uint32_t got = r ? __shfl_xor_sync(kFullMask, send, r) : send;
                    b0 = (from == 0) ? got : b0;
                    b1 = (from == 1) ? got : b1;
                    b2 = (from == 2) ? got : b2;
                    b3 = (from == 3) ? got : b3;
                }
                st_stream16(a.dst + (c0 + cb * 8 + g) * a.R + r0 + (rbg + kk) * 8, make_uint4(b0, b1, b2, b3));
            }
        } else {
            for (int idx = tid; idx < kTile * kTile; idx += kThreads) {
                const int ocl = idx / kTile, orow = idx % kTile;
                if (c0 + ocl < a.C && r0 + orow < a.R)
                    a.dst[(c0 + ocl) * a.R + r0 + orow] = sm[orow * 64 + (((ocl >> 3) ^ (orow & 7)) << 3) + (ocl & 7)];
            }
        }
        // every thread orders its reads of buffer s before the tensor copy
        // that refills it (the copy writes through the async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0 && a.issue_copies) {
            const int64_t tn = t + static_cast<int64_t>(kStages) * gridDim.x;
            if (tn < a.n_tiles) issue(s, tn);
        }
    }
}

__device__ __forceinline__ void stmatrix_x4(uint32_t addr, uint32_t d0, uint32_t d1, uint32_t d2, uint32_t d3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(d0), "r"(d1),
                 "r"(d2), "r"(d3)
                 : "memory");
}

constexpr int kOutBufs = 2;

// Both directions through the tensor-memory accelerator: the input tile
// arrives under the 128-byte swizzle, each warp transposes its 8 x 8 blocks
// with ldmatrix .trans and writes them with stmatrix into an output tile laid
// out under the same swizzle, and one thread stores that tile with a tensor
// copy.  Edge tiles need no special case: the load fills out-of-range
// elements with zeros and the store drops them.  Output buffers are double
// buffered; a buffer is rewritten only after the store issued from it two
// tiles earlier has finished reading it.
__global__ void __launch_bounds__(kThreads)
    transpose16_tma_ls_kernel(const __grid_constant__ CUtensorMap map_in, const __grid_constant__ CUtensorMap map_out,
                              const TmaArgs a) {
    pdl_launch_dependents();
    pdl_wait();  // before the first tensor copy
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[kStages];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t out_base = base + kStages * kTileBytes;
    const int tid = threadIdx.x;
    const uint32_t bar0 = smem_u32(&bars[0]);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8u * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    auto issue = [&](int s, int64_t t) {
        const int64_t tr = t / a.tiles_c, tc = t - tr * a.tiles_c;
        mbar_expect_tx(bar0 + 8u * s, kTileBytes);
        tma_load_2d(base + s * kTileBytes, &map_in, static_cast<int>(tc * kTile), static_cast<int>(tr * kTile),
                    bar0 + 8u * s);
    };
    if (tid == 0 && a.issue_copies) {
        for (int s = 0; s < kStages; ++s) {
            const int64_t t = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (t < a.n_tiles) issue(s, t);
        }
    }

    const int lane = tid & 31, warp = tid >> 5;
    const int m = lane >> 3, i8 = lane & 7;  // matrix addressed by this lane, its row
    for (int64_t it = 0;; ++it) {
        const int64_t t = blockIdx.x + it * gridDim.x;
        if (t >= a.n_tiles) break;
        const int s = static_cast<int>(it % kStages);
        const uint32_t ob = out_base + static_cast<uint32_t>(it & 1) * kTileBytes;
        const bool ok = mbar_wait_bounded(bar0 + 8u * s, static_cast<uint32_t>((it / kStages) & 1), a.wait_ns);
        if (tid == 0 && it >= kOutBufs) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicOr(a.status, 1u << SWZ_ERR_TIMEOUT);
            if (a.issue_copies) {
                for (int64_t j = it; j < it + kStages; ++j) {
                    const int64_t tj = blockIdx.x + j * gridDim.x;
                    if (tj >= a.n_tiles) break;
                    mbar_wait_bounded(bar0 + 8u * static_cast<uint32_t>(j % kStages),
                                      static_cast<uint32_t>((j / kStages) & 1), a.wait_ns);
                }
            }
            if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            return;
        }
        const uint32_t ib = base + s * kTileBytes;
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
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();  // output tile complete, input buffer s consumed
        if (tid == 0) {
            const int64_t tr = t / a.tiles_c, tc = t - tr * a.tiles_c;
            tma_store_2d(&map_out, static_cast<int>(tr * kTile), static_cast<int>(tc * kTile), ob);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            const int64_t tn = t + static_cast<int64_t>(kStages) * gridDim.x;
            if (a.issue_copies && tn < a.n_tiles) issue(s, tn);
        }
    }
    if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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

// The load+store kernel needs more than the default 48 KiB of dynamic shared
// memory; the attribute is set once per device.
bool ls_smem_attribute_set(int smem) {
    static std::mutex mu;
    static bool done[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        if (cudaFuncSetAttribute(transpose16_tma_ls_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return false;
        done[dev] = true;
    }
    return true;
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

    CUtensorMap map;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(R)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(C) * 2};
    const cuuint32_t box[2] = {kTile, kTile};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(src), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SWZ_ERR_CUDA;

    TmaArgs a;
    a.dst = static_cast<uint16_t *>(dst);
    a.R = R;
    a.C = C;
    a.tiles_c = (C + kTile - 1) / kTile;
    a.n_tiles = ((R + kTile - 1) / kTile) * a.tiles_c;
    a.vec_store_ok = ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) && (R % 8 == 0);
    a.issue_copies = issue_copies;
    a.wait_ns = wait_ns;
    a.status = status;
    int grid = sm_count() * 4;
    if (a.n_tiles < grid) grid = static_cast<int>(a.n_tiles);
    if (a.vec_store_ok) {
        // the output (C x R, rows of R elements) also goes out through a tensor map
        CUtensorMap map_out;
        const cuuint64_t odim[2] = {static_cast<cuuint64_t>(R), static_cast<cuuint64_t>(C)};
        const cuuint64_t ostride[1] = {static_cast<cuuint64_t>(R) * 2};
        if (encode(&map_out, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, dst, odim, ostride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SWZ_ERR_CUDA;
        const int smem = (kStages + kOutBufs) * kTileBytes + 1024;
        if (!ls_smem_attribute_set(smem)) return SWZ_ERR_CUDA;
        return launched(launch_pdl(transpose16_tma_ls_kernel, dim3(grid), dim3(kThreads), smem, st, map, map_out, a));
    }
    transpose16_tma_kernel<<<grid, kThreads, kStages * kTileBytes + 1024, st>>>(map, a);
    return launch_status();
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

    CUtensorMap map;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {kTile, kTile};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(src), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SWZ_ERR_CUDA;
    TmaArgs a;
    a.dst = static_cast<uint16_t *>(dst);
    a.R = rows;
    a.C = cols;
    a.tiles_c = (cols + kTile - 1) / kTile;
    a.n_tiles = ((rows + kTile - 1) / kTile) * a.tiles_c;
    a.vec_store_ok = ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) && (rows % 8 == 0);
    a.issue_copies = issue_copies;
    a.wait_ns = wait_ns;
    a.status = scratch;
    int grid = sm_count() * 4;
    if (a.n_tiles < grid) grid = static_cast<int>(a.n_tiles);
    transpose16_tma_kernel<<<grid, kThreads, kStages * kTileBytes + 1024, st>>>(map, a);
    const swz_status s = launch_status();
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
