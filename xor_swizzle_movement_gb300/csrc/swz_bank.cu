// swz_bank.cu -- shared-memory bank-conflict profiler for warp access
// patterns, and the batched slice collision (sm_103a).
//
// Model (see swz.h): 32 banks of 4 bytes; per pass, the cost is the largest
// number of distinct 4-byte words that fall in one bank; same-word lanes are
// served together.  Accesses of 8 bytes take two passes of 16 lanes, 16
// bytes four passes of 8 lanes; up to 4 bytes one pass of 32 lanes.
//
// One lane profiles whole patterns, two at a time.  Each warp stages 64
// consecutive patterns (8 KiB of addresses) in shared memory with cp.async,
// two batches in flight; a pattern's 128 bytes form one row, stored with its
// 16-byte chunks XOR-ed by the row index mod 8, so the copies into the row and
// each lane's reads of its own row are both free of bank conflicts.
//
// Aligned patterns (every active access on a multiple of its width, or a
// sub-word access inside one word): an access unit -- the word, or the
// W-byte chunk -- shares no word with another unit, so a pass costs the
// largest number of distinct units in one bank group.  The lane makes a key
// of each unit with the bank-group bits on top and the unit's other address
// bits below them.  Sorting a pass's keys (Batcher's odd-even merge network,
// all in registers) puts each group's units together and equal units side by
// side, and one scan counts the distinct keys of each group.  An inactive lane
// takes the address of the pass's first active lane, which adds nothing.  For
// addresses below 2^18 bytes (all of shared memory) a key fits in 16 bits and
// a lane sorts its two patterns side by side, two keys per word with 16-bit
// SIMD min and max; otherwise 32-bit keys, one pattern after the other.
// Every lane does the same work, so the warp never diverges on the data.
//
// A batch holding an unaligned pattern (one lane may then touch up to five
// words, and neighbours may share some of them) is counted on words instead:
// every word an active lane touches becomes a key, and a pass's keys (up to
// 64) are sorted and counted the same way.
#include "swz_common.cuh"

namespace swz {
namespace {

constexpr int kLaneWarps = 2;  // warps per CTA

template <int W>
struct Passes {
    static constexpr int n = W <= 4 ? 1 : W / 4;  // passes per access
    static constexpr int lanes = 32 / n;          // lanes per pass
};

// ---- one lane, one aligned pattern --------------------------------------------

__device__ __forceinline__ void order2(uint32_t &x, uint32_t &y) {
    const uint32_t lo = min(x, y);
    y = max(x, y);
    x = lo;
}

// The same on two 16-bit keys per word, each half on its own.
__device__ __forceinline__ void order2x(uint32_t &x, uint32_t &y) {
    uint32_t lo, hi;
    asm("min.u16x2 %0, %1, %2;" : "=r"(lo) : "r"(x), "r"(y));
    asm("max.u16x2 %0, %1, %2;" : "=r"(hi) : "r"(x), "r"(y));
    x = lo;
    y = hi;
}

template <bool PK>
__device__ __forceinline__ void order(uint32_t &x, uint32_t &y) {
    if constexpr (PK) order2x(x, y);
    else order2(x, y);
}

// Batcher's odd-even merge of k[LO .. LO+N), whose two halves are sorted,
// restricted to the elements LO, LO + R, LO + 2R, ...: merge the even and the
// odd subsequence (stride 2R), then order each odd element with the next one.
template <bool PK, int LO, int N, int R, int SZ>
__device__ __forceinline__ void oe_merge(uint32_t (&k)[SZ]) {
    if constexpr (2 * R < N) {
        oe_merge<PK, LO, N, 2 * R>(k);
        oe_merge<PK, LO + R, N, 2 * R>(k);
#pragma unroll
        for (int i = LO + R; i + R < LO + N; i += 2 * R) order<PK>(k[i], k[i + R]);
    } else {
        order<PK>(k[LO], k[LO + R]);
    }
}

// Sorts k[LO .. LO+N), N a power of two (19 / 63 / 191 / 543 compare-
// exchanges for 8 / 16 / 32 / 64 keys).  PK: two 16-bit keys per word,
// sorted side by side.
template <bool PK, int LO, int N, int SZ>
__device__ __forceinline__ void oe_sort(uint32_t (&k)[SZ]) {
    if constexpr (N > 1) {
        oe_sort<PK, LO, N / 2>(k);
        oe_sort<PK, LO + N / 2, N / 2>(k);
        oe_merge<PK, LO, N, 1>(k);
    }
}

// Sorts each pass's keys.
template <int W, bool PK>
__device__ __forceinline__ void sort_passes(uint32_t (&k)[32]) {
    if constexpr (Passes<W>::n == 1) {
        oe_sort<PK, 0, 32>(k);
    } else if constexpr (Passes<W>::n == 2) {
        oe_sort<PK, 0, 16>(k);
        oe_sort<PK, 16, 16>(k);
    } else {
        oe_sort<PK, 0, 8>(k);
        oe_sort<PK, 8, 8>(k);
        oe_sort<PK, 16, 8>(k);
        oe_sort<PK, 24, 8>(k);
    }
}

// Cost of the pattern in this lane's row (chunk c at row[c ^ sw]), m its
// active lanes, on 32-bit keys.  bad: some active access is unaligned; the
// result is then meaningless and the count on words (lane_words_cost) must
// replace it.
template <int W, bool MASKED>
__device__ __forceinline__ void lane_pattern_cost(const uint4 *row, int sw, uint32_t m, int &worst, int &total,
                                                  bool &bad) {
    constexpr int kPasses = Passes<W>::n, kLpp = Passes<W>::lanes;
    // keys of different bank groups differ in their top 5 / 4 / 3 bits
    constexpr uint32_t kNextGroup = 1u << (kPasses == 1 ? 27 : (kPasses == 2 ? 28 : 29));
    uint32_t k[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 v = row[c ^ sw];
        k[4 * c] = v.x;
        k[4 * c + 1] = v.y;
        k[4 * c + 2] = v.z;
        k[4 * c + 3] = v.w;
    }
    uint32_t mis = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        uint32_t u;
        if constexpr (W == 1) u = 0u;
        else if constexpr (W == 2) u = k[i] & (k[i] >> 1) & 1u;  // byte 3 of a word: the access straddles
        else u = k[i] & static_cast<uint32_t>(W - 1);
        if constexpr (MASKED) u = ((m >> i) & 1u) ? u : 0u;
        mis |= u;
        const uint32_t w = k[i] & ~3u;     // the unit's first byte (W >= 4 aligned: the address itself)
        k[i] = __funnelshift_r(w, w, 7);  // rotate right by 7: bank group on top
    }
    bad = mis != 0u;
    if constexpr (MASKED) {
#pragma unroll
        for (int q = 0; q < kPasses; ++q) {
            uint32_t kf = k[q * kLpp];
#pragma unroll
            for (int i = kLpp - 1; i >= 0; --i)
                if ((m >> (q * kLpp + i)) & 1u) kf = k[q * kLpp + i];
#pragma unroll
            for (int i = 0; i < kLpp; ++i)
                if (!((m >> (q * kLpp + i)) & 1u)) k[q * kLpp + i] = kf;
        }
    }
    sort_passes<W, false>(k);
    worst = 0;
    total = 0;
#pragma unroll
    for (int q = 0; q < kPasses; ++q) {
        int run = 1, mx = 1;  // distinct keys so far in the current group; the largest such count
#pragma unroll
        for (int i = 1; i < kLpp; ++i) {
            const uint32_t x = k[q * kLpp + i] ^ k[q * kLpp + i - 1];
            run = x >= kNextGroup ? 1 : run + (x != 0u ? 1 : 0);
            mx = max(mx, run);
        }
        uint32_t pm = m;
        if constexpr (kPasses > 1) pm = (m >> (q * kLpp)) & ((1u << kLpp) - 1u);
        const int cost = pm ? mx : 0;
        worst = max(worst, cost);
        total += cost;
    }
}

// Two patterns per lane on 16-bit keys: rows a and b (chunk c at a[c ^ sw]),
// active masks ma and mb.  A key is the bank-group bits of the unit's address
// (bits 2..6) over its bits 7..17, which holds every unit of an address below
// 2^18 bytes; ok is false when some address of either row is not below that,
// and the results are then not set.  Inactive lanes take the address of their
// pass's first active lane (0 when the pass has none).  bad[0], bad[1]: some
// active access of that row is unaligned.
template <int W, bool MASKED>
__device__ __forceinline__ void lane_pair_cost16(const uint4 *a, const uint4 *b, int sw, uint32_t ma, uint32_t mb,
                                                 int (&worst)[2], int (&total)[2], bool (&bad)[2], bool &ok) {
    constexpr int kPasses = Passes<W>::n, kLpp = Passes<W>::lanes;
    // 16-bit keys of different bank groups differ in their top 5 / 4 / 3 bits
    constexpr uint32_t kGroupBits = (kPasses == 1 ? 0xF800u : (kPasses == 2 ? 0xF000u : 0xE000u)) * 0x10001u;
    uint32_t fa[kPasses], fb[kPasses];  // first active address of each pass
    if constexpr (MASKED) {
#pragma unroll
        for (int q = 0; q < kPasses; ++q) {
            const uint32_t pa = kPasses == 1 ? ma : (ma >> (q * kLpp)) & ((1u << (kLpp & 31)) - 1u);
            const uint32_t pb = kPasses == 1 ? mb : (mb >> (q * kLpp)) & ((1u << (kLpp & 31)) - 1u);
            const int ia = q * kLpp + __ffs(pa) - 1, ib = q * kLpp + __ffs(pb) - 1;
            fa[q] = pa ? reinterpret_cast<const uint32_t *>(a)[((ia >> 2) ^ sw) * 4 + (ia & 3)] : 0u;
            fb[q] = pb ? reinterpret_cast<const uint32_t *>(b)[((ib >> 2) ^ sw) * 4 + (ib & 3)] : 0u;
        }
    }
    uint32_t k[32];
    uint32_t acc_a = 0, acc_b = 0;  // OR of the addresses (W = 2: of a & (a >> 1))
    uint32_t hi = 0;                // OR of both rows' addresses, for the range
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 va = a[c ^ sw], vb = b[c ^ sw];
        const uint32_t xa[4] = {va.x, va.y, va.z, va.w}, xb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = 4 * c + j;
            uint32_t ua = xa[j], ub = xb[j];
            if constexpr (MASKED) {
                ua = (ma & (1u << i)) ? ua : fa[i / kLpp];
                ub = (mb & (1u << i)) ? ub : fb[i / kLpp];
            }
            if constexpr (W >= 4) {
                acc_a |= ua;
                acc_b |= ub;
            } else {
                hi |= ua | ub;
                if constexpr (W == 2) {
                    acc_a |= ua & (ua >> 1);
                    acc_b |= ub & (ub >> 1);
                }
            }
            // word indices of a (low half) and b (high half), each rotated left by
            // 11 within its half: bank group (bits 2..6) over address bits 7..17
            const uint32_t wp = __byte_perm(ua >> 2, ub >> 2, 0x5410);
            k[i] = ((wp << 11) & 0xF800F800u) | ((wp >> 5) & 0x07FF07FFu);
        }
    }
    if constexpr (W >= 4) hi = acc_a | acc_b;
    constexpr uint32_t kMis = W == 1 ? 0u : (W == 2 ? 1u : static_cast<uint32_t>(W - 1));
    bad[0] = (acc_a & kMis) != 0u;
    bad[1] = (acc_b & kMis) != 0u;
    ok = (hi >> 18) == 0u;
    if (!__all_sync(kFullMask, ok)) return;  // some lane needs 32-bit keys: the warp takes them
    sort_passes<W, true>(k);
    worst[0] = worst[1] = total[0] = total[1] = 0;
#pragma unroll
    for (int q = 0; q < kPasses; ++q) {
        // per half: distinct keys so far in the current group, and the largest such count
        uint32_t run = 0x00010001u, mx = 0x00010001u;
#pragma unroll
        for (int i = 1; i < kLpp; ++i) {
            const uint32_t x = k[q * kLpp + i] ^ k[q * kLpp + i - 1];
            uint32_t d, g;
            asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(0x00010001u));               // a new key
            asm("min.u16x2 %0, %1, %2;" : "=r"(g) : "r"(x & kGroupBits), "r"(0x00010001u));  // a new group
            const uint32_t msk = g * 0xFFFFu;  // 0xFFFF in the halves where a group starts
            run = ((run + d) & ~msk) | (0x00010001u & msk);
            asm("max.u16x2 %0, %1, %2;" : "=r"(mx) : "r"(mx), "r"(run));
        }
        const uint32_t pa = kPasses == 1 ? ma : (ma >> (q * kLpp)) & ((1u << (kLpp & 31)) - 1u);
        const uint32_t pb = kPasses == 1 ? mb : (mb >> (q * kLpp)) & ((1u << (kLpp & 31)) - 1u);
        const int ca = pa ? static_cast<int>(mx & 0xFFFFu) : 0, cb = pb ? static_cast<int>(mx >> 16) : 0;
        worst[0] = max(worst[0], ca);
        total[0] += ca;
        worst[1] = max(worst[1], cb);
        total[1] += cb;
    }
}

// Any pattern, aligned or not: every word an active lane touches (first ..
// last, the last repeated to fill J slots) becomes a key with its bank on top
// and its other bits below, and a pass's keys (padded to 64 with copies of its
// first key) are sorted and counted as above.  PK: rows a and b side by side
// on 16-bit keys, which hold words below 2^16; returns false, setting nothing,
// when some lane's row reaches 2^18 - 16 bytes (the warp then takes 32-bit
// keys, one row at a time: PK false, row a only, results in worst[0] and
// total[0]).  Inactive lanes take the address of their pass's first active lane.
template <int W, bool MASKED, bool PK>
__device__ __forceinline__ bool lane_words_cost(const uint4 *a, const uint4 *b, int sw, uint32_t ma, uint32_t mb,
                                                int (&worst)[2], int (&total)[2]) {
    constexpr int kPasses = Passes<W>::n, kLpp = Passes<W>::lanes;
    constexpr int J = W <= 4 ? 2 : (W == 8 ? 3 : 5);  // most words one access touches
    constexpr int kChunks = kLpp / 4;                  // 16-byte chunks of addresses per pass
    const uint32_t m[2] = {ma, mb};
    const uint4 *row[2] = {a, b};
    constexpr int kRowsHere = PK ? 2 : 1;
    if constexpr (PK) {
        uint32_t hi = 0;  // every address below 2^18 - 16: no a + W - 1 wraps, no word + 4 leaves its half
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v = row[h][c ^ sw];
                const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t u = (!MASKED || (m[h] & (1u << (4 * c + j)))) ? x[j] : 0u;
                    hi |= u | (u + 16u);
                }
            }
        if (!__all_sync(kFullMask, (hi >> 18) == 0u)) return false;
    }
    worst[0] = worst[1] = total[0] = total[1] = 0;
#pragma unroll 1
    for (int q = 0; q < kPasses; ++q) {
        uint32_t pm[2], f[2];  // the pass's active lanes and first active address per row
#pragma unroll
        for (int h = 0; h < kRowsHere; ++h) {
            pm[h] = kPasses == 1 ? m[h] : (m[h] >> (q * kLpp)) & ((1u << (kLpp & 31)) - 1u);
            f[h] = 0u;
            if constexpr (MASKED) {
                const int i = q * kLpp + __ffs(pm[h]) - 1;
                if (pm[h]) f[h] = reinterpret_cast<const uint32_t *>(row[h])[((i >> 2) ^ sw) * 4 + (i & 3)];
            }
        }
        uint32_t k[64];
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            uint32_t x[2][4];
#pragma unroll
            for (int h = 0; h < kRowsHere; ++h) {
                const uint4 v = row[h][(q * kChunks + c) ^ sw];
                x[h][0] = v.x;
                x[h][1] = v.y;
                x[h][2] = v.z;
                x[h][3] = v.w;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = 4 * c + j;  // lane within the pass
                if constexpr (PK) {
                    uint32_t u[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) u[h] = (!MASKED || (pm[h] & (1u << i))) ? x[h][j] : f[h];
                    const uint32_t w0 = __byte_perm(u[0] >> 2, u[1] >> 2, 0x5410);
                    const uint32_t wl = __byte_perm((u[0] + (W - 1)) >> 2, (u[1] + (W - 1)) >> 2, 0x5410);
#pragma unroll
                    for (int t = 0; t < J; ++t) {
                        uint32_t w;  // word t of the access, or its last word
                        asm("min.u16x2 %0, %1, %2;" : "=r"(w) : "r"(w0 + t * 0x00010001u), "r"(wl));
                        k[i * J + t] = ((w << 11) & 0xF800F800u) | ((w >> 5) & 0x07FF07FFu);
                    }
                } else {
                    const uint32_t u = (!MASKED || (pm[0] & (1u << i))) ? x[0][j] : f[0];
                    const uint32_t w0 = u >> 2;
                    const uint32_t wl = static_cast<uint32_t>((static_cast<uint64_t>(u) + (W - 1)) >> 2);  // <= 2^30
#pragma unroll
                    for (int t = 0; t < J; ++t) {
                        const uint32_t w = min(w0 + t, wl);
                        k[i * J + t] = ((w & 31u) << 27) | (w >> 5);
                    }
                }
            }
        }
#pragma unroll
        for (int i = kLpp * J; i < 64; ++i) k[i] = k[0];
        oe_sort<PK, 0, 64>(k);
        int cost[2];
        if constexpr (PK) {
            uint32_t run = 0x00010001u, mx = 0x00010001u;
#pragma unroll
            for (int i = 1; i < 64; ++i) {
                const uint32_t x = k[i] ^ k[i - 1];
                uint32_t d, g;
                asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(0x00010001u));
                asm("min.u16x2 %0, %1, %2;" : "=r"(g) : "r"(x & 0xF800F800u), "r"(0x00010001u));
                const uint32_t msk = g * 0xFFFFu;
                run = ((run + d) & ~msk) | (0x00010001u & msk);
                asm("max.u16x2 %0, %1, %2;" : "=r"(mx) : "r"(mx), "r"(run));
            }
            cost[0] = static_cast<int>(mx & 0xFFFFu);
            cost[1] = static_cast<int>(mx >> 16);
        } else {
            int run = 1, mx = 1;
#pragma unroll
            for (int i = 1; i < 64; ++i) {
                const uint32_t x = k[i] ^ k[i - 1];
                run = x >= (1u << 27) ? 1 : run + (x != 0u ? 1 : 0);
                mx = max(mx, run);
            }
            cost[0] = mx;
        }
#pragma unroll
        for (int h = 0; h < kRowsHere; ++h) {
            const int c = pm[h] ? cost[h] : 0;
            worst[h] = max(worst[h], c);
            total[h] += c;
        }
    }
    return true;
}

// ---- kernel ---------------------------------------------------------------------

constexpr int kRows = 64;  // patterns per warp and batch: two per lane

struct __align__(16) LaneStage {
    uint4 rows[2][kRows * 8];  // two batches of 64 rows of 8 chunks; chunk c of row r at r * 8 + (c ^ (r & 7))
    uint32_t mask[2][kRows];
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// W = access bytes per lane (1, 2, 4, 8, 16); MASKED: an active-lane mask per
// pattern; VEC: the address array is 16-byte aligned and rows are copied in
// 16-byte chunks (otherwise word by word).  Each warp takes batches of 64
// patterns at a grid stride; lane l profiles rows l and l + 32 of a batch.
template <int W, bool MASKED, bool VEC>
__global__ void __launch_bounds__(kLaneWarps * 32, 6)  // 6 CTAs (12 warps, 198 KiB of stages) per SM
    bank_profile_kernel(const uint32_t *__restrict__ addrs, const uint32_t *__restrict__ active, int64_t n,
                        int32_t *__restrict__ ways, int32_t *__restrict__ wavefronts) {
    __shared__ LaneStage s_stage[kLaneWarps];
    pdl_launch_dependents();
    pdl_wait();  // before any global memory access
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    LaneStage &st = s_stage[wid];
    const int64_t n_batches = (n + kRows - 1) / kRows;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kLaneWarps;
    auto stage = [&](int64_t b, int buf) {
        if (b < n_batches) {
            const int64_t p0 = b * kRows;
            if constexpr (VEC) {
#pragma unroll
                for (int j = 0; j < kRows / 4; ++j) {
                    const int r = 4 * j + (lane >> 3), c = lane & 7;
                    if (p0 + r < n) cp_async16(&st.rows[buf][r * 8 + (c ^ (r & 7))], addrs + (p0 + r) * 32 + c * 4);
                }
            } else {
                const int c = lane >> 2;
                for (int r = 0; r < kRows && p0 + r < n; ++r)
                    cp_async4(reinterpret_cast<uint32_t *>(&st.rows[buf][r * 8 + (c ^ (r & 7))]) + (lane & 3),
                              addrs + (p0 + r) * 32 + lane);
            }
            if constexpr (MASKED) {
                if (p0 + lane < n) cp_async4(&st.mask[buf][lane], active + p0 + lane);
                if (p0 + 32 + lane < n) cp_async4(&st.mask[buf][32 + lane], active + p0 + 32 + lane);
            }
        }
        cp_async_commit();
    };
    int64_t b = static_cast<int64_t>(blockIdx.x) * kLaneWarps + wid;
    stage(b, 0);
    for (int buf = 0; b < n_batches; b += stride, buf ^= 1) {
        stage(b + stride, buf ^ 1);
        cp_async_wait_1();
        __syncwarp();  // every lane's copies of this batch are visible to the warp
        const int64_t p[2] = {b * kRows + lane, b * kRows + 32 + lane};
        const uint32_t m[2] = {MASKED ? st.mask[buf][lane] : kFullMask, MASKED ? st.mask[buf][32 + lane] : kFullMask};
        const uint4 *row[2] = {&st.rows[buf][lane * 8], &st.rows[buf][(32 + lane) * 8]};
        int worst[2], total[2];
        bool bad[2], ok;
        lane_pair_cost16<W, MASKED>(row[0], row[1], lane & 7, m[0], m[1], worst, total, bad, ok);
        if (!__all_sync(kFullMask, ok)) {  // an address at or above 2^18: 32-bit keys, one row at a time
#pragma unroll 1  // one copy of the 32-bit path: fewer registers
            for (int h = 0; h < 2; ++h) lane_pattern_cost<W, MASKED>(row[h], lane & 7, m[h], worst[h], total[h], bad[h]);
        }
        if constexpr (W > 1) {  // a 1-byte access never straddles a word
            if (__any_sync(kFullMask, (bad[0] && p[0] < n) || (bad[1] && p[1] < n))) {
                // an unaligned pattern in the batch: word keys for all of it
                if (!lane_words_cost<W, MASKED, true>(row[0], row[1], lane & 7, m[0], m[1], worst, total)) {
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        int w1[2], t1[2];
                        lane_words_cost<W, MASKED, false>(row[h], row[h], lane & 7, m[h], 0u, w1, t1);
                        worst[h] = w1[0];
                        total[h] = t1[0];
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (p[h] < n) {
                ways[p[h]] = worst[h];
                wavefronts[p[h]] = total[h];
            }
        }
        __syncwarp();  // the warp is done with this buffer before it is staged again
    }
    cp_async_wait_all();
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

template <int W, bool MASKED>
static cudaError_t launch_profile(bool vec, unsigned grid, cudaStream_t st, const uint32_t *addrs,
                                  const uint32_t *active, int64_t n, int32_t *ways, int32_t *wavefronts) {
    const dim3 g(grid), blk(kLaneWarps * 32);
    return vec ? launch_pdl(bank_profile_kernel<W, MASKED, true>, g, blk, 0, st, addrs, active, n, ways, wavefronts)
               : launch_pdl(bank_profile_kernel<W, MASKED, false>, g, blk, 0, st, addrs, active, n, ways, wavefronts);
}

template <int W>
static cudaError_t launch_profile(bool vec, unsigned grid, cudaStream_t st, const uint32_t *addrs,
                                  const uint32_t *active, int64_t n, int32_t *ways, int32_t *wavefronts) {
    return active ? launch_profile<W, true>(vec, grid, st, addrs, active, n, ways, wavefronts)
                  : launch_profile<W, false>(vec, grid, st, addrs, active, n, ways, wavefronts);
}

swz_status bank_profile_launch(const uint32_t *addrs, const uint32_t *active, int64_t n, int width,
                               int32_t *ways, int32_t *wavefronts, cudaStream_t st) {
    const int64_t batches = (n + kRows - 1) / kRows;  // 64 patterns per warp
    int64_t grid = (batches + kLaneWarps - 1) / kLaneWarps;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 6;  // one wave of resident CTAs, then a grid stride
    if (grid > cap) grid = cap;
    const unsigned g = static_cast<unsigned>(grid);
    const bool vec = (reinterpret_cast<uintptr_t>(addrs) & 15u) == 0;
    cudaError_t e;
    switch (width) {
        case 1: e = launch_profile<1>(vec, g, st, addrs, active, n, ways, wavefronts); break;
        case 2: e = launch_profile<2>(vec, g, st, addrs, active, n, ways, wavefronts); break;
        case 4: e = launch_profile<4>(vec, g, st, addrs, active, n, ways, wavefronts); break;
        case 8: e = launch_profile<8>(vec, g, st, addrs, active, n, ways, wavefronts); break;
        case 16: e = launch_profile<16>(vec, g, st, addrs, active, n, ways, wavefronts); break;
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
