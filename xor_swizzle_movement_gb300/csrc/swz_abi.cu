// swz_abi.cu -- the C ABI declared in include/swz.h: argument validation,
// dispatch to the kernels, status codes.  Nothing here allocates memory.
#include "swz_common.cuh"

#include <atomic>
#include <cstdio>

namespace swz {

swz_status relayout_launch(void *dst, const void *src, int64_t n_tiles, int64_t tile_elems, int esize,
                           int B, int M, int S, int direction, cudaStream_t st);
swz_status relayout_tma_launch(void *dst, const void *src, int64_t n_tiles, int64_t tile_elems, int esize,
                               int B, int M, int S, int direction, cudaStream_t st);
int relayout_tma_path(const void *dst, const void *src, int64_t n_tiles, int64_t tile_elems, int esize, int B,
                      int M, int S);
swz_status transpose_launch(void *dst, const void *src, int64_t R, int64_t C, int esize, int variant,
                            cudaStream_t st);
swz_status transpose_relayout_launch(void *dst, const void *src, int64_t R, int64_t C, int esize, int64_t te,
                                     int B, int M, int S, cudaStream_t st);
swz_status bank_profile_launch(const uint32_t *addrs, const uint32_t *active, int64_t n, int width,
                               int32_t *ways, int32_t *wavefronts, cudaStream_t st);
swz_status slice_collision_launch(const uint64_t *A, int64_t n, int B, int M, int S, uint64_t *C,
                                  cudaStream_t st);

swz_status launch_status() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SWZ_OK : SWZ_ERR_CUDA;
}

swz_status launched(cudaError_t launch_result) {
    if (launch_result != cudaSuccess) {
        cudaGetLastError();  // clear it: the status carries it
        return SWZ_ERR_CUDA;
    }
    return launch_status();
}

// Streaming multiprocessors of the current device, queried once per device
// and cached (launch geometry is sized in multiples of it).  Returns 1 if the
// query fails; the launch that follows then reports the error.
int sm_count() {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    if (dev >= 0 && dev < kMaxDevices) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 1;
    }
    if (dev >= 0 && dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

// L2 cache size of the current device in bytes, queried once per device and
// cached.  Returns 0 if the query fails (every buffer then counts as larger).
int64_t l2_bytes() {
    constexpr int kMaxDevices = 64;
    static std::atomic<int64_t> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < kMaxDevices) {
        const int64_t c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

bool host_resident(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}

bool ranges_overlap(const void *a, int64_t a_bytes, const void *b, int64_t b_bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

namespace {

bool valid_esize(int e) { return e == 1 || e == 2 || e == 4 || e == 8 || e == 16; }

// B, M, S in element units.  S = 0 makes the map non-injective; negative S
// puts the read field at M and the written one |S| bits above it (sw_fwd).
bool valid_bms(int B, int M, int S, int max_total) {
    if (B < 0 || B > 16 || M < 0 || M > 32 || S < -32 || S > 32) return false;
    if (B == 0) return true;  // the identity
    const int a = S < 0 ? -S : S;
    return a >= 1 && B + M + a <= max_total;
}

// a * b without int64 overflow (a, b >= 0)
bool mul_ok(int64_t a, int64_t b, int64_t *out) {
    if (a != 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}

bool aligned_to(const void *p, int64_t n) { return (reinterpret_cast<uintptr_t>(p) % static_cast<uintptr_t>(n)) == 0; }

}  // namespace
}  // namespace swz

namespace swz {
namespace {
// Validation shared by the relayout entry points; *launch is set when there
// is work to launch (tile_elems then holds rows * cols).
swz_status check_relayout(void *dst, const void *src, int64_t n_tiles, int64_t rows, int64_t cols, int esize, int B,
                          int M, int S, int direction, int64_t *tile_elems, bool *launch) {
    *launch = false;
    if (!valid_esize(esize) || !valid_bms(B, M, S, 48) || (direction != 0 && direction != 1))
        return SWZ_ERR_PARAM;
    if (n_tiles < 0 || rows < 0 || cols < 0) return SWZ_ERR_SHAPE;
    int64_t n_elems, n_bytes;
    if (!mul_ok(rows, cols, tile_elems) || !mul_ok(n_tiles, *tile_elems, &n_elems) ||
        !mul_ok(n_elems, esize, &n_bytes))
        return SWZ_ERR_SHAPE;
    if (n_elems == 0) return SWZ_OK;
    if (*tile_elems % (int64_t(1) << (B ? sw_write_hi(B, M, S) : M)) != 0) return SWZ_ERR_SHAPE;
    if (!dst || !src) return SWZ_ERR_NULL;
    if (!aligned_to(dst, esize) || !aligned_to(src, esize)) return SWZ_ERR_ALIGN;
    if (ranges_overlap(dst, n_bytes, src, n_bytes)) return SWZ_ERR_ALIAS;
    *launch = true;
    return SWZ_OK;
}
}  // namespace
}  // namespace swz

extern "C" {

swz_status swz_relayout(void *dst, const void *src, int64_t n_tiles, int64_t rows, int64_t cols,
                        int esize, int B, int M, int S, int direction, void *stream) {
    using namespace swz;
    int64_t tile_elems = 0;
    bool launch = false;
    const swz_status v = check_relayout(dst, src, n_tiles, rows, cols, esize, B, M, S, direction, &tile_elems, &launch);
    if (v != SWZ_OK || !launch) return v;
    return relayout_launch(dst, src, n_tiles, tile_elems, esize, B, M, S, direction,
                           static_cast<cudaStream_t>(stream));
}

swz_status swz_relayout_tma(void *dst, const void *src, int64_t n_tiles, int64_t rows, int64_t cols,
                            int esize, int B, int M, int S, int direction, void *stream) {
    using namespace swz;
    int64_t tile_elems = 0;
    bool launch = false;
    const swz_status v = check_relayout(dst, src, n_tiles, rows, cols, esize, B, M, S, direction, &tile_elems, &launch);
    if (v != SWZ_OK || !launch) return v;
    return relayout_tma_launch(dst, src, n_tiles, tile_elems, esize, B, M, S, direction,
                               static_cast<cudaStream_t>(stream));
}

int swz_relayout_tma_path(const void *dst, const void *src, int64_t n_tiles, int64_t rows, int64_t cols, int esize,
                          int B, int M, int S, int direction) {
    using namespace swz;
    int64_t tile_elems = 0;
    bool launch = false;
    const swz_status v = check_relayout(const_cast<void *>(dst), src, n_tiles, rows, cols, esize, B, M, S, direction,
                                        &tile_elems, &launch);
    if (v != SWZ_OK) return -static_cast<int>(v);
    if (!launch) return 0;
    return relayout_tma_path(dst, src, n_tiles, tile_elems, esize, B, M, S);
}

swz_status swz_transpose(void *dst, const void *src, int64_t rows, int64_t cols, int esize, int variant,
                         void *stream) {
    using namespace swz;
    if (!valid_esize(esize) || variant < SWZ_T_SWIZZLED || variant > SWZ_T_TMA) return SWZ_ERR_PARAM;
    if (variant == SWZ_T_TMA && esize != 2) return SWZ_ERR_PARAM;
    if (rows < 0 || cols < 0) return SWZ_ERR_SHAPE;
    int64_t n_elems, n_bytes;
    if (!mul_ok(rows, cols, &n_elems) || !mul_ok(n_elems, esize, &n_bytes)) return SWZ_ERR_SHAPE;
    if (n_elems == 0) return SWZ_OK;
    if (!dst || !src) return SWZ_ERR_NULL;
    if (!aligned_to(dst, esize) || !aligned_to(src, esize)) return SWZ_ERR_ALIGN;
    if (ranges_overlap(dst, n_bytes, src, n_bytes)) return SWZ_ERR_ALIAS;
    return transpose_launch(dst, src, rows, cols, esize, variant, static_cast<cudaStream_t>(stream));
}

swz_status swz_transpose_relayout(void *dst, const void *src, int64_t rows, int64_t cols, int esize,
                                  int64_t tile_elems, int B, int M, int S, void *stream) {
    using namespace swz;
    if (!valid_esize(esize) || !valid_bms(B, M, S, 48)) return SWZ_ERR_PARAM;
    if (rows < 0 || cols < 0 || tile_elems <= 0) return SWZ_ERR_SHAPE;
    int64_t n_elems, n_bytes;
    if (!mul_ok(rows, cols, &n_elems) || !mul_ok(n_elems, esize, &n_bytes)) return SWZ_ERR_SHAPE;
    if (n_elems % tile_elems != 0 || tile_elems % (int64_t(1) << (B ? sw_write_hi(B, M, S) : M)) != 0)
        return SWZ_ERR_SHAPE;
    if (n_elems == 0) return SWZ_OK;
    if (!dst || !src) return SWZ_ERR_NULL;
    if (!aligned_to(dst, esize) || !aligned_to(src, esize)) return SWZ_ERR_ALIGN;
    if (ranges_overlap(dst, n_bytes, src, n_bytes)) return SWZ_ERR_ALIAS;
    return transpose_relayout_launch(dst, src, rows, cols, esize, tile_elems, B, M, S,
                                     static_cast<cudaStream_t>(stream));
}

swz_status swz_bank_profile(const uint32_t *byte_addrs, const uint32_t *active, int64_t n,
                            int access_bytes, int32_t *ways, int32_t *wavefronts, void *stream) {
    using namespace swz;
    if (!valid_esize(access_bytes)) return SWZ_ERR_PARAM;
    if (n < 0 || n > INT64_MAX / 128) return SWZ_ERR_SHAPE;
    if (n == 0) return SWZ_OK;
    if (!byte_addrs || !ways || !wavefronts) return SWZ_ERR_NULL;
    if (!aligned_to(byte_addrs, 4) || !aligned_to(ways, 4) || !aligned_to(wavefronts, 4) ||
        (active && !aligned_to(active, 4)))
        return SWZ_ERR_ALIGN;
    return bank_profile_launch(byte_addrs, active, n, access_bytes, ways, wavefronts,
                               static_cast<cudaStream_t>(stream));
}

swz_status swz_slice_collision(uint64_t A, int B, int M, int S, uint64_t *C_out) {
    using namespace swz;
    if (!valid_bms(B, M, S, 64)) return SWZ_ERR_PARAM;
    if (!C_out) return SWZ_ERR_NULL;
    *C_out = A & ~sw_fwd(A, B, M, S);
    return SWZ_OK;
}

swz_status swz_slice_layout(uint64_t A, int B, int M, int S, uint64_t *strides, int *n_bits) {
    using namespace swz;
    if (!valid_bms(B, M, S, 64)) return SWZ_ERR_PARAM;
    if (!strides || !n_bits) return SWZ_ERR_NULL;
    if ((A & ~sw_fwd(A, B, M, S)) != 0) return SWZ_ERR_UNSUPPORTED;
    int k = 0;
    for (int bit = 0; bit < 64; ++bit)
        if ((A >> bit) & 1u) strides[k++] = sw_fwd(uint64_t(1) << bit, B, M, S);
    *n_bits = k;
    return SWZ_OK;
}

swz_status swz_slice_collision_batch(const uint64_t *A, int64_t n, int B, int M, int S, uint64_t *C,
                                     void *stream) {
    using namespace swz;
    if (!valid_bms(B, M, S, 64)) return SWZ_ERR_PARAM;
    if (n < 0 || n > INT64_MAX / 8) return SWZ_ERR_SHAPE;
    if (n == 0) return SWZ_OK;
    if (!A || !C) return SWZ_ERR_NULL;
    if (!aligned_to(A, 8) || !aligned_to(C, 8)) return SWZ_ERR_ALIGN;
    if (ranges_overlap(A, n * 8, C, n * 8) && A != C) return SWZ_ERR_ALIAS;
    return slice_collision_launch(A, n, B, M, S, C, static_cast<cudaStream_t>(stream));
}

int64_t swz_layout_text(char *buf, int64_t cap, int64_t rows, int64_t cols, int esize, int B, int M, int S) {
    using namespace swz;
    int64_t n_elems;
    if (rows < 0 || cols < 0 || esize < 1 || cap < 0 || (cap > 0 && !buf) || !valid_bms(B, M, S, 64) ||
        !mul_ok(rows, cols, &n_elems))
        return -1;
    int64_t len = 0;
    auto put = [&](const char *text, int n) {
        for (int i = 0; i < n; ++i, ++len)
            if (len < cap - 1) buf[len] = text[i];
    };
    char cell[48];
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            const uint64_t phys = sw_fwd(static_cast<uint64_t>(r * cols + c), B, M, S);
            const uint64_t bank = (phys * static_cast<uint64_t>(esize) / 4) % 32;
            const int n = snprintf(cell, sizeof cell, c ? " %llu/%llu" : "%llu/%llu",
                                   static_cast<unsigned long long>(phys), static_cast<unsigned long long>(bank));
            put(cell, n);
        }
        put("\n", 1);
    }
    if (cap > 0) buf[len < cap - 1 ? len : cap - 1] = '\0';
    return len;
}

uint64_t swz_apply(uint64_t x, int B, int M, int S) {
    if (!swz::valid_bms(B, M, S, 64)) return x;
    return swz::sw_fwd(x, B, M, S);
}

const char *swz_status_string(int status) {
    switch (status) {
        case SWZ_OK: return "SWZ_OK";
        case SWZ_ERR_NULL: return "SWZ_ERR_NULL: a required pointer is NULL";
        case SWZ_ERR_PARAM: return "SWZ_ERR_PARAM: swizzle parameter, element size, direction or variant out of range";
        case SWZ_ERR_SHAPE: return "SWZ_ERR_SHAPE: bad sizes or a tile not closed under the swizzle";
        case SWZ_ERR_ALIGN: return "SWZ_ERR_ALIGN: pointer not aligned to the element size";
        case SWZ_ERR_ALIAS: return "SWZ_ERR_ALIAS: dst and src overlap";
        case SWZ_ERR_CUDA: return "SWZ_ERR_CUDA: CUDA launch error";
        case SWZ_ERR_TIMEOUT: return "SWZ_ERR_TIMEOUT: a bounded device wait gave up";
        case SWZ_ERR_UNSUPPORTED: return "SWZ_ERR_UNSUPPORTED: no kernel for this request";
        default: return "unknown swz_status";
    }
}

int swz_version(void) { return 100; }

}  // extern "C"
