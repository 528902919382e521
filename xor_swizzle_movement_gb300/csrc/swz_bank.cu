// swz_bank.cu -- shared-memory bank-conflict profiler for warp access
// patterns, one warp per pattern (sm_103a).
//
// Model (see swz.h): 32 banks of 4 bytes; per pass, the cost is the largest
// number of distinct 4-byte words that fall in one bank; same-word lanes are
// served together.  Accesses of 8 bytes take two passes of 16 lanes, 16
// bytes four passes of 8 lanes; up to 4 bytes one pass of 32 lanes.
//
// Lane l of the warp holds lane l's address, so the pattern is read with one
// coalesced 128-byte load.  Aligned patterns (the only ones real hardware
// accepts: a w-byte access on a multiple of w, or a sub-word access that does
// not straddle a word) are counted with two warp matches: the first keeps one
// lane per distinct (pass, access unit), the second groups those leaders by
// (pass, bank group) and its population count is the number of distinct
// words in that bank.  Unaligned patterns, where one lane may touch up to
// five words and neighbours may share some of them, are counted exactly with
// a per-warp table in shared memory.
#include "swz_common.cuh"

namespace swz {
namespace {

constexpr int kWarpsPerCta = 8;

__device__ __forceinline__ int reduce_max_segment(int v, int seg) {
    // max over aligned groups of `seg` lanes (seg = 8, 16 or 32)
    for (int o = 1; o < seg; o <<= 1) v = max(v, __shfl_xor_sync(kFullMask, v, o));
    return v;
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
    bank_profile_kernel(const uint32_t *__restrict__ addrs, const uint32_t *__restrict__ active,
                        int64_t n, int width, int32_t *__restrict__ ways,
                        int32_t *__restrict__ wavefronts) {
    __shared__ uint32_t s_first[kWarpsPerCta][32];
    __shared__ int s_nw[kWarpsPerCta][32];
    __shared__ int s_cnt[kWarpsPerCta][4][32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int passes = width <= 4 ? 1 : width / 4;
    const int lpp = 32 / passes;  // lanes per pass
    const int pass = lane / lpp;
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + wid; p < n; p += warps_total) {
        const uint32_t a = __ldcs(addrs + p * 32 + lane);
        const uint32_t mask = active ? __ldcs(active + p) : kFullMask;
        const bool on = (mask >> lane) & 1u;
        const bool aligned = width <= 4 ? ((a & 3u) + static_cast<uint32_t>(width) <= 4u)
                                        : ((a & static_cast<uint32_t>(width - 1)) == 0u);
        int cost;  // cost of this lane's pass, valid on every lane of the pass
        if (__all_sync(kFullMask, !on || aligned)) {
            const uint32_t unit_bytes = width <= 4 ? 4u : static_cast<uint32_t>(width);
            const uint32_t unit = a / unit_bytes;               // access unit (word or w-byte chunk)
            const uint32_t groups = 32u / (unit_bytes / 4u);    // bank groups of unit_bytes
            const unsigned long long solo = (1ull << 63) | static_cast<unsigned long long>(lane);
            const unsigned long long k1 =
                on ? ((static_cast<unsigned long long>(pass) << 40) | unit) : solo;
            const unsigned m1 = __match_any_sync(kFullMask, k1);
            const bool leader = on && (__ffs(m1) - 1 == lane);
            const unsigned long long k2 =
                leader ? ((static_cast<unsigned long long>(pass) << 40) | (unit % groups)) : solo;
            const unsigned m2 = __match_any_sync(kFullMask, k2);
            cost = reduce_max_segment(leader ? __popc(m2) : 0, lpp);
        } else {
            // exact count: candidate words first .. first + nw - 1 per lane
            const unsigned long long last = (static_cast<unsigned long long>(a) + width - 1) >> 2;
            const uint32_t first = a >> 2;
            const int nw = on ? static_cast<int>(last - first + 1) : 0;
            s_first[wid][lane] = first;
            s_nw[wid][lane] = nw;
#pragma unroll
            for (int q = 0; q < 4; ++q) s_cnt[wid][q][lane] = 0;
            __syncwarp();
            for (int i = 0; i < 5; ++i) {
                const bool valid = i < nw;
                const unsigned long long wd = static_cast<unsigned long long>(first) + i;
                const unsigned long long key =
                    valid ? ((static_cast<unsigned long long>(pass) << 40) | wd)
                          : ((1ull << 63) | static_cast<unsigned long long>(lane));
                const unsigned m = __match_any_sync(kFullMask, key);
                bool fresh = valid && (__ffs(m) - 1 == lane);
                if (fresh && i > 0) {
                    // did a lane of this pass touch the same word in an earlier round?
                    for (int l2 = pass * lpp; l2 < (pass + 1) * lpp; ++l2) {
                        const long long d = static_cast<long long>(wd) - static_cast<long long>(s_first[wid][l2]);
                        if (d >= 0 && d < i && d < s_nw[wid][l2]) fresh = false;
                    }
                }
                if (fresh) atomicAdd(&s_cnt[wid][pass][static_cast<int>(wd & 31u)], 1);
            }
            __syncwarp();
            int mine = 0;
            for (int q = 0; q < passes; ++q) {
                const int c = reduce_max_segment(s_cnt[wid][q][lane], 32);
                if (q == pass) mine = c;
            }
            cost = mine;
            __syncwarp();
        }
        // one representative lane per pass carries that pass's cost
        int worst = (lane % lpp == 0) ? cost : 0;
        int total = worst;
        for (int o = 1; o < 32; o <<= 1) {
            worst = max(worst, __shfl_xor_sync(kFullMask, worst, o));
            total += __shfl_xor_sync(kFullMask, total, o);
        }
        if (lane == 0) {
            ways[p] = worst;
            wavefronts[p] = total;
        }
    }
}

__global__ void slice_collision_kernel(const uint64_t *__restrict__ A, int64_t n, int B, int M,
                                       int S, uint64_t *__restrict__ C) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint64_t a = A[i];
        C[i] = a & ~sw_fwd(a, B, M, S);
    }
}

}  // namespace

swz_status bank_profile_launch(const uint32_t *addrs, const uint32_t *active, int64_t n, int width,
                               int32_t *ways, int32_t *wavefronts, cudaStream_t st) {
    int64_t grid = (n + kWarpsPerCta - 1) / kWarpsPerCta;
    if (grid > 152LL * 64) grid = 152LL * 64;  // grid-stride beyond 64 CTAs per SM
    bank_profile_kernel<<<static_cast<unsigned>(grid), kWarpsPerCta * 32, 0, st>>>(addrs, active, n, width,
                                                                                ways, wavefronts);
    return launch_status();
}

swz_status slice_collision_launch(const uint64_t *A, int64_t n, int B, int M, int S, uint64_t *C,
                                  cudaStream_t st) {
    int64_t grid = (n + 255) / 256;
    if (grid > 152LL * 16) grid = 152LL * 16;
    slice_collision_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(A, n, B, M, S, C);
    return launch_status();
}

}  // namespace swz
