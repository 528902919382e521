// swz_common.cuh -- device helpers shared by the swizzle kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "swz.h"

namespace swz {

constexpr unsigned kFullMask = 0xffffffffu;

// Swizzle<B,M,S> on an element offset: one shift, one mask, one XOR.
// ("CuTe Swizzle 学习手册", section "Swizzle 数学公式".)
__host__ __device__ __forceinline__ uint64_t sw_fwd(uint64_t x, int B, int M, int S) {
    const uint64_t mask = (B >= 64) ? ~0ull : ((1ull << B) - 1ull);
    return x ^ (((x >> (M + S)) & mask) << M);
}

// Inverse of sw_fwd.  For S >= B the function is an involution and one step
// suffices.  For 1 <= S < B the read field overlaps the written one; writing
// y = x ^ f(x), the iteration x <- y ^ f(x) started at x = y fixes S more bits
// of x per step from the top of the written field downwards, so ceil(B / S)
// steps reach the exact inverse.
__host__ __device__ __forceinline__ uint64_t sw_inv(uint64_t y, int B, int M, int S, int steps) {
    const uint64_t mask = (B >= 64) ? ~0ull : ((1ull << B) - 1ull);
    uint64_t x = y;
    for (int i = 0; i < steps; ++i) x = y ^ (((x >> (M + S)) & mask) << M);
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

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

}  // namespace swz

// Host-side helpers shared by the launchers (defined in swz_abi.cu).
namespace swz {
swz_status launch_status();
bool ranges_overlap(const void *a, int64_t a_bytes, const void *b, int64_t b_bytes);
}  // namespace swz
