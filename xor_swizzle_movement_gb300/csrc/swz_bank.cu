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
// not straddle a word) are counted in claim rounds through a 32-slot per-warp
// table (one slot per pass and bank group): a round costs one shared store,
// one shared load and a ballot, and a pass takes exactly as many rounds as
// its cost.  (Two warp-wide match instructions per pattern, the obvious
// alternative, cost about 50 SM cycles each here.)  Unaligned patterns, where
// one lane may touch up to five words and neighbours may share some of them,
// are counted exactly with a per-warp table of word candidates.
#include "swz_common.cuh"

namespace swz {
namespace {

constexpr int kWarpsPerCta = 8;

// W = access bytes per lane (1, 2, 4, 8, 16)
template <int W>
__global__ void __launch_bounds__(kWarpsPerCta * 32, 8)  // 8 CTAs (64 warps) per SM: 32 registers
    bank_profile_kernel(const uint32_t *__restrict__ addrs, const uint32_t *__restrict__ active,
                        int64_t n, int32_t *__restrict__ ways, int32_t *__restrict__ wavefronts) {
    constexpr int kPasses = W <= 4 ? 1 : W / 4;
    constexpr int kLpp = 32 / kPasses;                       // lanes per pass
    constexpr uint32_t kUnitShift = W <= 4 ? 2 : (W == 8 ? 3 : 4);  // log2 of the access unit (>= a word)
    __shared__ uint32_t s_tab[kWarpsPerCta][32];
    __shared__ uint32_t s_first[kWarpsPerCta][32];
    __shared__ int s_nw[kWarpsPerCta][32];
    __shared__ int s_cnt[kWarpsPerCta][4][32];
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int pass = lane / kLpp;
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + wid; p < n; p += warps_total) {
        const uint32_t a = __ldcs(addrs + p * 32 + lane);
        const uint32_t mask = active ? __ldcs(active + p) : kFullMask;
        const bool on = (mask >> lane) & 1u;
        const bool aligned = W <= 4 ? ((a & 3u) + static_cast<uint32_t>(W) <= 4u)
                                    : ((a & static_cast<uint32_t>(W - 1)) == 0u);
        int cost;  // cost of this lane's pass, valid on every lane of the pass
        if (__all_sync(kFullMask, !on || aligned)) {
            // An aligned access unit (a word, or a W-byte chunk) never shares a
            // word with a different unit, so the pass cost is the largest
            // number of distinct units in one bank group.  Count it by rounds:
            // every lane still waiting writes its unit into its group's slot,
            // one write per slot wins, and every lane whose unit is the one in
            // its slot is served.  Each round serves exactly one distinct unit
            // per slot, so a pass takes as many rounds as its worst group holds
            // distinct units.
            const uint32_t unit = a >> kUnitShift;
            const int slot = pass * kLpp + static_cast<int>(unit & static_cast<uint32_t>(kLpp - 1));
            const unsigned pass_lanes = (kLpp == 32) ? kFullMask : (((1u << (kLpp & 31)) - 1u) << (pass * kLpp));
            volatile uint32_t *tab = s_tab[wid];
            unsigned rem = __ballot_sync(kFullMask, on);
            int rounds = 0;
            while (rem) {  // warp-uniform; every round serves at least one lane
                const bool waiting = (rem >> lane) & 1u;
                if (waiting) tab[slot] = unit;
                __syncwarp();
                const bool served = waiting && tab[slot] == unit;
                __syncwarp();
                rounds += (rem & pass_lanes) != 0u;
                rem &= ~__ballot_sync(kFullMask, served);
            }
            cost = rounds;
        } else {
            // exact count: candidate words first .. first + nw - 1 per lane
            const unsigned long long last = (static_cast<unsigned long long>(a) + W - 1) >> 2;
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
                    for (int l2 = pass * kLpp; l2 < (pass + 1) * kLpp; ++l2) {
                        const long long d = static_cast<long long>(wd) - static_cast<long long>(s_first[wid][l2]);
                        if (d >= 0 && d < i && d < s_nw[wid][l2]) fresh = false;
                    }
                }
                if (fresh) atomicAdd(&s_cnt[wid][pass][static_cast<int>(wd & 31u)], 1);
            }
            __syncwarp();
            int mine = 0;
#pragma unroll
            for (int q = 0; q < kPasses; ++q) {
                const int c = static_cast<int>(__reduce_max_sync(kFullMask, static_cast<unsigned>(s_cnt[wid][q][lane])));
                if (q == pass) mine = c;
            }
            cost = mine;
            __syncwarp();
        }
        unsigned worst, total;
        if constexpr (kPasses == 1) {
            worst = total = static_cast<unsigned>(cost);  // already uniform across the warp
        } else {
            // one representative lane per pass carries that pass's cost
            const unsigned rep = (lane % kLpp == 0) ? static_cast<unsigned>(cost) : 0u;
            worst = __reduce_max_sync(kFullMask, rep);
            total = __reduce_add_sync(kFullMask, rep);
        }
        if (lane == 0) {
            ways[p] = static_cast<int32_t>(worst);
            wavefronts[p] = static_cast<int32_t>(total);
        }
    }
}

// Element by element (A or C not 16-byte aligned, and the odd last mask).
__global__ void slice_collision_kernel(const uint64_t *A, int64_t i0, int64_t n, int B, int M, int S,
                                       uint64_t *C) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = i0 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint64_t a = A[i];
        C[i] = a & ~sw_fwd(a, B, M, S);
    }
}

// Two masks per 16-byte access, four accesses in flight per thread, one CTA
// per 1024 accesses.  Plain loads (not the read-only path): A and C may be the
// same array.
__global__ void __launch_bounds__(256) slice_collision_vec_kernel(const ulonglong2 *A, int64_t npairs, int B,
                                                                  int M, int S, ulonglong2 *C) {
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * 4 + threadIdx.x;
    ulonglong2 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t i = base + static_cast<int64_t>(k) * blockDim.x;
        if (i < npairs) v[k] = A[i];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t i = base + static_cast<int64_t>(k) * blockDim.x;
        if (i < npairs) {
            ulonglong2 c;
            c.x = v[k].x & ~sw_fwd(v[k].x, B, M, S);
            c.y = v[k].y & ~sw_fwd(v[k].y, B, M, S);
            C[i] = c;
        }
    }
}

}  // namespace

swz_status bank_profile_launch(const uint32_t *addrs, const uint32_t *active, int64_t n, int width,
                               int32_t *ways, int32_t *wavefronts, cudaStream_t st) {
    int64_t grid = (n + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 64;  // grid-stride beyond 64 CTAs per SM
    if (grid > cap) grid = cap;
    const unsigned g = static_cast<unsigned>(grid);
    cudaError_t e;
    switch (width) {
        case 1: e = launch_pdl(bank_profile_kernel<1>, dim3(g), dim3(kWarpsPerCta * 32), 0, st, addrs, active, n, ways, wavefronts); break;
        case 2: e = launch_pdl(bank_profile_kernel<2>, dim3(g), dim3(kWarpsPerCta * 32), 0, st, addrs, active, n, ways, wavefronts); break;
        case 4: e = launch_pdl(bank_profile_kernel<4>, dim3(g), dim3(kWarpsPerCta * 32), 0, st, addrs, active, n, ways, wavefronts); break;
        case 8: e = launch_pdl(bank_profile_kernel<8>, dim3(g), dim3(kWarpsPerCta * 32), 0, st, addrs, active, n, ways, wavefronts); break;
        case 16: e = launch_pdl(bank_profile_kernel<16>, dim3(g), dim3(kWarpsPerCta * 32), 0, st, addrs, active, n, ways, wavefronts); break;
        default: return SWZ_ERR_PARAM;
    }
    return launched(e);
}

swz_status slice_collision_launch(const uint64_t *A, int64_t n, int B, int M, int S, uint64_t *C,
                                  cudaStream_t st) {
    const bool aligned16 = ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(C)) & 15u) == 0;
    int64_t done = 0;  // masks handled by the vector kernel
    if (aligned16 && n >= 2) {
        const int64_t npairs = n / 2;
        const int64_t grid = (npairs + 1023) / 1024;
        if (grid > 0x7fffffffLL) return SWZ_ERR_SHAPE;
        const swz_status s = launched(launch_pdl(slice_collision_vec_kernel, dim3(static_cast<unsigned>(grid)),
                                                 dim3(256), 0, st, reinterpret_cast<const ulonglong2 *>(A), npairs,
                                                 B, M, S, reinterpret_cast<ulonglong2 *>(C)));
        if (s != SWZ_OK) return s;
        done = 2 * npairs;
    }
    if (done == n) return SWZ_OK;
    int64_t grid = (n - done + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
    if (grid > cap) grid = cap;
    return launched(launch_pdl(slice_collision_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st, A, done,
                               n, B, M, S, C));
}

}  // namespace swz
