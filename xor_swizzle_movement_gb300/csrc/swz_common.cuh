// swz_common.cuh -- device helpers shared by the swizzle kernels (sm_103a).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "swz.h"

namespace swz {

constexpr unsigned kFullMask = 0xffffffffu;

// The two B-bit fields of Swizzle<B,M,S>.  S > 0: the written field (ZZZ)
// starts at bit M and the read field (YYY) S bits above it ("CuTe Swizzle
// 学习手册", section "Swizzle 数学公式").  S < 0: YYY is moved leftward onto
// ZZZ ("NVIDIA CuTe Swizzle", the bit-diagram comment), so the read field
// starts at M and the written one |S| bits above it; the lowest M bits stay
// out of the map either way.
__host__ __device__ __forceinline__ int sw_read_lo(int M, int S) { return S > 0 ? M + S : M; }
__host__ __device__ __forceinline__ int sw_write_lo(int M, int S) { return S > 0 ? M : M - S; }
// Bit above the written field: offsets close under the swizzle in aligned
// blocks of 2^sw_write_hi elements.
__host__ __device__ __forceinline__ int sw_write_hi(int B, int M, int S) { return sw_write_lo(M, S) + B; }
// Steps of sw_inv that reach the exact inverse (see there).
__host__ __device__ __forceinline__ int sw_inv_steps(int B, int S) {
    const int a = S < 0 ? -S : S;
    return (B > 0 && a < B) ? (B + a - 1) / a : 1;
}

// Swizzle<B,M,S> on an element offset: one shift, one mask, one XOR.
__host__ __device__ __forceinline__ uint64_t sw_fwd(uint64_t x, int B, int M, int S) {
    const uint64_t mask = (B >= 64) ? ~0ull : ((1ull << B) - 1ull);
    return x ^ (((x >> sw_read_lo(M, S)) & mask) << sw_write_lo(M, S));
}

// Inverse of sw_fwd.  For |S| >= B the function is an involution and one
// step suffices.  For 1 <= |S| < B the read field overlaps the written one;
// writing y = x ^ f(x), the iteration x <- y ^ f(x) started at x = y fixes
// |S| more bits of x per step (from the top of the written field downwards
// for S > 0, from its bottom upwards for S < 0), so ceil(B / |S|) steps reach
// the exact inverse.
__host__ __device__ __forceinline__ uint64_t sw_inv(uint64_t y, int B, int M, int S, int steps) {
    const uint64_t mask = (B >= 64) ? ~0ull : ((1ull << B) - 1ull);
    const int r = sw_read_lo(M, S), w = sw_write_lo(M, S);
    uint64_t x = y;
    for (int i = 0; i < steps; ++i) x = y ^ (((x >> r) & mask) << w);
    return x;
}

// Streaming 16-byte global access.  Loads bypass L1 (the data is touched once).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// An L2 policy with the default eviction priority.
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// An L2 policy that marks lines as first to evict: for data read once.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint4 ld_stream16_hint(const void *p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ void st_stream16(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// A 16-byte store under an L2 policy (l2_evict_first_policy: for output that
// nothing reads soon; l2_evict_normal_policy: as a plain store).
__device__ __forceinline__ void st_hint16(void *p, uint4 v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w), "l"(policy)
                 : "memory");
}

// The same store marked streaming (st.global.cs): its line leaves L2 first.
// For output that nothing reads soon and that could not stay in L2 anyway;
// output that a following launch reads from L2 keeps the plain store.
__device__ __forceinline__ void st_once16(void *p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Programmatic dependent launch.  A kernel launched with the
// programmatic-stream-serialization attribute may start while the previous
// kernel on its stream is still running; pdl_wait() blocks until that kernel
// has completed and its writes are visible, so it must precede every global
// memory access (reads of its results and writes it might still read).
// pdl_launch_dependents() lets the next such kernel start launching; called on
// entry, it lets the next grid fill SMs during this grid's last wave.  Both
// are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}


// 16-byte vectors of E-byte elements: V lanes, log2 V.
template <int E>
struct VecTraits {
    static constexpr int V = 16 / E;  // lanes (elements) per vector
    static constexpr int LV = (E == 1) ? 4 : (E == 2) ? 3 : (E == 4) ? 2 : (E == 8) ? 1 : 0;
};

// out lane l = in lane l ^ L
template <int E>
__device__ __forceinline__ uint4 lanes_xor(uint4 v, uint32_t L) {
    if constexpr (E == 16) {
        return v;
    } else {
        uint32_t wx;
        if constexpr (E == 8) wx = L << 1;
        else if constexpr (E == 4) wx = L;
        else if constexpr (E == 2) wx = L >> 1;
        else wx = L >> 2;
        uint32_t w0 = v.x, w1 = v.y, w2 = v.z, w3 = v.w, t;
        if (wx & 1u) { t = w0; w0 = w1; w1 = t; t = w2; w2 = w3; w3 = t; }
        if (wx & 2u) { t = w0; w0 = w2; w2 = t; t = w1; w1 = w3; w3 = t; }
        if constexpr (E == 2) {
            if (L & 1u) {
                w0 = __byte_perm(w0, 0, 0x1032); w1 = __byte_perm(w1, 0, 0x1032);
                w2 = __byte_perm(w2, 0, 0x1032); w3 = __byte_perm(w3, 0, 0x1032);
            }
        }
        if constexpr (E == 1) {
            const uint32_t sel = 0x3210u ^ (0x1111u * (L & 3u));
            w0 = __byte_perm(w0, 0, sel); w1 = __byte_perm(w1, 0, sel);
            w2 = __byte_perm(w2, 0, sel); w3 = __byte_perm(w3, 0, sel);
        }
        return make_uint4(w0, w1, w2, w3);
    }
}

// A fixed permutation of the 16 bytes of v: output byte 4w + i comes from the
// input byte the host encoded in sel[3w .. 3w + 2] (two prmt pick from the low
// and the high 8 bytes, a third merges them).
__device__ __forceinline__ uint4 bytes_permute(uint4 v, const uint32_t *sel) {
    uint32_t o[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t lo = __byte_perm(v.x, v.y, sel[3 * w]);
        const uint32_t hi = __byte_perm(v.z, v.w, sel[3 * w + 1]);
        o[w] = __byte_perm(lo, hi, sel[3 * w + 2]);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}


// Host side: the prmt selectors that make bytes_permute move lane l of a
// 16-byte vector of esize-byte elements from lane src_lane[l].
inline void lane_map_selectors(const int *src_lane, int esize, uint32_t sel[12]) {
    int src_byte[16];
    const int lanes = 16 / esize;
    for (int l = 0; l < lanes; ++l)
        for (int bb = 0; bb < esize; ++bb) src_byte[l * esize + bb] = src_lane[l] * esize + bb;
    for (int w = 0; w < 4; ++w) {
        uint32_t s_lo = 0, s_hi = 0, s_mix = 0;
        for (int i = 0; i < 4; ++i) {
            const int sb = src_byte[4 * w + i];
            if (sb < 8) {
                s_lo |= static_cast<uint32_t>(sb) << (4 * i);
                s_mix |= static_cast<uint32_t>(i) << (4 * i);
            } else {
                s_hi |= static_cast<uint32_t>(sb - 8) << (4 * i);
                s_mix |= static_cast<uint32_t>(4 + i) << (4 * i);
            }
        }
        sel[3 * w] = s_lo;
        sel[3 * w + 1] = s_hi;
        sel[3 * w + 2] = s_mix;
    }
}
}  // namespace swz

// Launch `kernel` with programmatic dependent launch allowed (see pdl_wait),
// or, with pdl false, as a plain launch (its pdl_wait is then a no-op).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_if(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
    return launch_pdl_if(true, kernel, grid, block, smem, st, std::forward<Args>(args)...);
}

// Host-side helpers shared by the launchers (defined in swz_abi.cu).
namespace swz {
swz_status launch_status();
swz_status launched(cudaError_t launch_result);  // status of a launch_pdl call
bool ranges_overlap(const void *a, int64_t a_bytes, const void *b, int64_t b_bytes);
int sm_count();  // SMs of the current device (cached per device)
int64_t l2_bytes();  // L2 cache bytes of the current device (cached per device)
bool host_resident(const void *p);  // p is host memory (pinned or pageable), not device or managed memory
}  // namespace swz
