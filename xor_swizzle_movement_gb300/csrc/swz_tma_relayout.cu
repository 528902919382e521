// swz_tma_relayout.cu -- relayout through the tensor-memory accelerator's
// hardware swizzle (sm_103a).
//
// A TMA tensor copy in the 32-, 64- or 128-byte swizzle mode XORs bits
// [4, 4 + B) of the shared-memory byte address with bits [7, 7 + B), B = 1, 2,
// 3: the byte-address Swizzle<B,4,3>, i.e. element Swizzle<B, 4 - log2 e, 3> on
// e-byte elements ("CuTe Swizzle 学习手册", sections "Sw<3,4,3> vs Sw<3,3,3>"
// and "H100 TMA + Swizzle").  The buffer is viewed as rows of 2^(B+4) bytes
// (the swizzle span) and moved in 8 KiB chunks:
//   forward  dst[sw(i)] = src[i]: a swizzled tensor load, then a plain bulk store;
//   inverse  dst[i] = src[sw(i)]: a plain bulk load, then a swizzled tensor store.
// Each chunk covers whole swizzle periods (2^(B+7) bytes) of whole tiles, so
// the tile-local swizzle equals the swizzle of the chunk-local offset.  One
// thread per CTA drives a ring of four 8 KiB buffers; every copy is
// asynchronous and every mbarrier wait is bounded (kWaitLimitNs) with the
// expiry recorded in the per-device status word.
#include "swz_tma_common.cuh"

namespace swz {

swz_status relayout_launch(void *dst, const void *src, int64_t n_tiles, int64_t tile_elems, int esize, int B,
                           int M, int S, int direction, cudaStream_t st);

namespace {

constexpr int kChunk = 8192;     // bytes per copy
constexpr int kRing = 4;         // buffers per CTA
constexpr int kCtasPerSm = 6;    // 33 KiB of shared memory each

struct TmaRelayoutArgs {
    uint8_t *dst;
    const uint8_t *src;
    int64_t bytes;          // the whole buffer
    int64_t n_chunks;
    int rows_per_chunk;     // kChunk / swizzle span
    int direction;
    uint64_t wait_ns;
    uint32_t *status;
};

__global__ void __launch_bounds__(32)
    relayout_tma_kernel(const __grid_constant__ CUtensorMap map, const TmaRelayoutArgs a) {
    pdl_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[kRing];
    if (threadIdx.x != 0) return;  // one thread issues every copy
    pdl_wait();                    // before the first copy
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // the swizzle is computed from address bits
    const uint32_t bar0 = smem_u32(&bars[0]);
    for (int s = 0; s < kRing; ++s) mbar_init(bar0 + 8u * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");

    auto chunk_bytes = [&](int64_t c) -> uint32_t {
        const int64_t left = a.bytes - c * kChunk;
        return static_cast<uint32_t>(left < kChunk ? left : kChunk);
    };
    auto issue_load = [&](int s, int64_t c) {
        const uint32_t buf = base + s * kChunk, bar = bar0 + 8u * s;
        if (a.direction == 0) {
            // a tensor box always transfers its full size (rows past the end are zero-filled)
            mbar_expect_tx(bar, kChunk);
            tma_load_2d(buf, &map, 0, static_cast<int>(c * a.rows_per_chunk), bar);
        } else {
            const uint32_t nb = chunk_bytes(c);
            mbar_expect_tx(bar, nb);
            bulk_load(buf, a.src + c * kChunk, nb, bar);
        }
    };
    auto issue_store = [&](int s, int64_t c) {
        const uint32_t buf = base + s * kChunk;
        if (a.direction == 0) bulk_store(a.dst + c * kChunk, buf, chunk_bytes(c));
        else tma_store_2d(&map, 0, static_cast<int>(c * a.rows_per_chunk), buf);  // rows past the end are dropped
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    };

    for (int s = 0; s < kRing; ++s) {
        const int64_t c = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
        if (c < a.n_chunks) issue_load(s, c);
    }
    for (int64_t it = 0;; ++it) {
        const int64_t c = blockIdx.x + it * gridDim.x;
        if (c >= a.n_chunks) break;
        const int s = static_cast<int>(it % kRing);
        if (!mbar_wait_bounded(bar0 + 8u * s, static_cast<uint32_t>((it / kRing) & 1), a.wait_ns)) {
            atomicOr(a.status, 1u << SWZ_ERR_TIMEOUT);
            // let the loads still in flight land before the CTA exits: those of
            // iterations it .. it + kRing - 1 (before the first refill) or
            // it .. it + kRing - 2 (after it)
            const int64_t last = it == 0 ? kRing - 1 : it + kRing - 2;
            for (int64_t j = it; j <= last; ++j) {
                if (blockIdx.x + j * gridDim.x >= a.n_chunks) break;
                mbar_wait_bounded(bar0 + 8u * static_cast<uint32_t>(j % kRing),
                                  static_cast<uint32_t>((j / kRing) & 1), a.wait_ns);
            }
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            return;
        }
        issue_store(s, c);
        if (it >= 1) {
            // the previous chunk's store has read its buffer: refill that buffer
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            const int64_t cn = c - gridDim.x + static_cast<int64_t>(kRing) * gridDim.x;
            if (cn < a.n_chunks) issue_load(static_cast<int>((it - 1) % kRing), cn);
        }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace

// Arguments are validated by the caller (swz_relayout_tma in swz_abi.cu).
swz_status relayout_tma_launch(void *dst, const void *src, int64_t n_tiles, int64_t tile_elems, int esize, int B,
                               int M, int S, int direction, cudaStream_t st) {
    int k = 0;
    while ((1 << k) < esize) ++k;
    const int64_t span = int64_t(16) << B;       // swizzle span: 32, 64 or 128 bytes
    const int64_t period = span * 8;             // 2^(B+7) bytes
    const int64_t tile_bytes = tile_elems * esize;
    const int64_t bytes = n_tiles * tile_bytes;
    const bool aligned = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
    EncodeTiledFn encode = encode_fn();
    const bool hw_mode = B >= 1 && B <= 3 && S == 3 && M + k == 4;
    if (!hw_mode || !aligned || !encode || tile_bytes % period != 0 || bytes / span >= (int64_t(1) << 31))
        return relayout_launch(dst, src, n_tiles, tile_elems, esize, B, M, S, direction, st);
    uint32_t *status = device_status_word(true);
    if (!status) return SWZ_ERR_CUDA;

    static const CUtensorMapSwizzle modes[4] = {CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                                                CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_SWIZZLE_128B};
    CUtensorMap map;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(span), static_cast<cuuint64_t>(bytes / span)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(span)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(span), static_cast<cuuint32_t>(kChunk / span)};
    const cuuint32_t estride[2] = {1, 1};
    void *tensor_side = direction == 0 ? const_cast<void *>(src) : dst;
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, tensor_side, gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, modes[B], CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SWZ_ERR_CUDA;

    TmaRelayoutArgs a;
    a.dst = static_cast<uint8_t *>(dst);
    a.src = static_cast<const uint8_t *>(src);
    a.bytes = bytes;
    a.n_chunks = (bytes + kChunk - 1) / kChunk;
    a.rows_per_chunk = static_cast<int>(kChunk / span);
    a.direction = direction;
    a.wait_ns = kWaitLimitNs;
    a.status = status;
    int64_t grid = 152LL * kCtasPerSm;
    if (a.n_chunks < grid) grid = a.n_chunks;
    return launched(launch_pdl(relayout_tma_kernel, dim3(static_cast<unsigned>(grid)), dim3(32), kRing * kChunk + 1024,
                               st, map, a));
}

}  // namespace swz
