/*
 * swz.h -- C ABI of the XOR-swizzle data-movement library for GB300 (sm_103a).
 *
 * The swizzle is CuTe's Swizzle<B, M, S> acting on an element offset x:
 *
 *     sw(x) = x ^ (((x >> (M + S)) & ((1 << B) - 1)) << M)
 *
 * ("CuTe Swizzle 学习手册", section "Swizzle 数学公式"; the same function with
 * base = M, bits = B, shift = S in "CUDA 013 - Swizzle 的工作原理", section
 * "计算公式").  The B bits that start at bit M + S are XOR-ed into the B bits
 * that start at bit M; the low M bits (a group of 2^M elements that stays
 * contiguous) and every other bit are kept.  All B, M, S arguments below are
 * in ELEMENT-offset units.
 *
 * A negative S moves the read field (YYY) leftward onto the written one
 * (ZZZ): the B bits that start at bit M are XOR-ed into the B bits that start
 * at bit M + |S|, i.e. sw(x) = x ^ (((x >> M) & ((1 << B) - 1)) << (M - S)).
 * ("NVIDIA CuTe Swizzle", the bit-diagram comment: the sign of SShift gives
 * the direction the YYY mask moves, and the low MBase bits stay constant.  The
 * pages give no formula for this case; this placement is the one that keeps
 * the low M bits out of the map, as for S > 0.)
 *
 * Conventions shared by every entry point:
 *   - Pointers named dst/src/out are DEVICE pointers owned by the caller (the
 *     relayout also accepts host memory the device can address); the library
 *     never allocates, frees or retains them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  GPU work is enqueued on it and the call returns without
 *     waiting; the caller synchronises.
 *   - The return value reports argument validation and launch errors only.
 *     On any error nothing is launched and no output byte is written.  A
 *     fault during execution surfaces, as in any CUDA call, at the next
 *     synchronising call on that stream.
 *   - No exception or C++ type crosses this boundary.
 */
#ifndef SWZ_H
#define SWZ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum swz_status {
    SWZ_OK = 0,
    SWZ_ERR_NULL = 1,        /* a required pointer is NULL */
    SWZ_ERR_PARAM = 2,       /* B, M, S, element size, direction or variant out of range */
    SWZ_ERR_SHAPE = 3,       /* negative or overflowing sizes, tile not closed under sw */
    SWZ_ERR_ALIGN = 4,       /* a pointer is not aligned to the element size */
    SWZ_ERR_ALIAS = 5,       /* dst and src overlap (in-place is not supported) */
    SWZ_ERR_CUDA = 6,        /* the CUDA runtime reported an error at launch */
    SWZ_ERR_TIMEOUT = 7,     /* a bounded device wait gave up (see swz_transpose) */
    SWZ_ERR_UNSUPPORTED = 8  /* a valid request the library has no kernel for */
} swz_status;

/* Transpose staging variants (see swz_transpose). */
enum {
    SWZ_T_SWIZZLED = 0,   /* shared-memory tile under the per-size swizzle */
    SWZ_T_UNSWIZZLED = 1, /* plain [T][T] tile: column access is bank-conflicted */
    SWZ_T_PADDED = 2,     /* [T][T + pad] tile: conflict-free, wastes shared memory */
    SWZ_T_TMA = 3         /* 16-bit data only: tile loaded by a TMA tensor copy
                             with the hardware 128-byte swizzle (and stored by
                             one when the output rows are whole 16-byte
                             vectors) */
};

/*
 * Batched tile relayout.
 *
 * Source: "CUDA 013 - Swizzle 的工作原理", sections "更通用的映射规则" and
 * "使用示例" (an element whose logical offset is o lives at the swizzled
 * offset sw(o)); "NVIDIA CuTe Swizzle" and "cutlass 入门" for the parameters.
 *
 * dst, src : buffers of n_tiles * rows * cols elements of esize bytes, each
 *            tile stored contiguously, row-major (offset o = r * cols + c).
 *            Normally device memory; host memory the device can address
 *            (pinned, or any on systems with address translation) also works,
 *            at the host link's rate.  A call with a host-resident buffer
 *            runs a grid sized for the link (4 CTAs per SM), so a relayout
 *            that reads host memory and one that writes it, on two streams,
 *            run at the same time and use both directions of the link.
 *            Pointers need only be aligned to esize; pointers off 16-byte
 *            alignment keep 16-byte global accesses (aligned chunks shifted
 *            in registers or staged in shared memory) at some cost in speed.
 * esize    : 1, 2, 4, 8 or 16 bytes.  Elements are copied as raw bits.
 * B, M, S  : swizzle parameters in element units; 0 <= B <= 16,
 *            0 <= M <= 32, -32 <= S <= 32, and when B > 0: S != 0 and
 *            B + M + |S| <= 48.  S = 0 is rejected (it is not a bijection);
 *            1 <= |S| < B is accepted (a bijection, but not its own
 *            inverse).  B = 0 is the identity.
 * direction: 0 = forward, logical row-major to swizzled physical order:
 *                dst[t][sw(i)] = src[t][i];
 *            1 = inverse, swizzled physical to logical:
 *                dst[t][i] = src[t][sw(i)].
 *            Offsets i are local to each tile.
 *
 * Errors: SWZ_ERR_NULL (dst or src NULL with a non-empty request),
 * SWZ_ERR_PARAM, SWZ_ERR_SHAPE (negative sizes, byte size overflowing
 * int64, or rows * cols not a multiple of 2^h, h the bit above the written
 * field: M + B for S > 0, M + |S| + B for S < 0, so that a tile would not be
 * closed under sw), SWZ_ERR_ALIGN (dst or src not aligned to esize),
 * SWZ_ERR_ALIAS (the two byte ranges overlap), SWZ_ERR_CUDA.
 * An empty request (no element) returns SWZ_OK and launches nothing.
 */
swz_status swz_relayout(void *dst, const void *src, int64_t n_tiles, int64_t rows,
                        int64_t cols, int esize, int B, int M, int S, int direction,
                        void *stream);

/*
 * Batched tile relayout through the tensor-memory accelerator's hardware
 * swizzle.
 *
 * Source: the TMA usage of "CuTe Swizzle 学习手册", sections "Sw<3,4,3> vs
 * Sw<3,3,3>" (Sw<3,4,3> is the 128-byte pattern the TMA descriptor carries)
 * and "H100 TMA + Swizzle".  The TMA 32-, 64- and 128-byte swizzle modes are
 * the byte-address Swizzle<1,4,3>, <2,4,3> and <3,4,3>, i.e. element
 * Swizzle<B, 4 - log2(esize), 3> for B = 1, 2, 3; the 128-byte mode with
 * 32-byte atoms is the byte-address Swizzle<2,5,2>, element
 * Swizzle<2, 5 - log2(esize), 2>.
 *
 * Same arguments, rules, errors and result as swz_relayout.  The swizzled side
 * of the copy runs on the TMA (a swizzled tensor load into shared memory, then
 * 16-byte stores of it in order; each mode is its own inverse, so both
 * directions are this copy) when (B, M + log2(esize), S) is one of the four
 * modes above, each tile holds a whole number of the mode's periods
 * (2^(B + M + log2(esize) + S) bytes) and dst and src are 16-byte aligned;
 * any other request runs swz_relayout's kernels (swz_relayout_tma_path tells
 * which).  The TMA
 * path's bounded waits report to swz_device_status() (its status word is the
 * one SWZ_T_TMA allocates on first use).
 */
swz_status swz_relayout_tma(void *dst, const void *src, int64_t n_tiles, int64_t rows,
                            int64_t cols, int esize, int B, int M, int S, int direction,
                            void *stream);

/*
 * The path swz_relayout_tma takes for these arguments, without running it:
 *   0  swz_relayout's register kernels;
 *   1  the TMA 32-byte mode (byte-address Swizzle<1,4,3>);
 *   2  the 64-byte mode (Swizzle<2,4,3>);
 *   3  the 128-byte mode (Swizzle<3,4,3>);
 *   4  the 128-byte mode with 32-byte atoms (Swizzle<2,5,2>);
 *  -s  the swz_status s that swz_relayout_tma would return for bad arguments.
 * An empty request returns 0.  Host function; pointers are not dereferenced.
 */
int swz_relayout_tma_path(const void *dst, const void *src, int64_t n_tiles, int64_t rows,
                          int64_t cols, int esize, int B, int M, int S, int direction);

/*
 * Matrix transpose HBM -> shared memory -> HBM.
 *
 * out[c][r] = in[r][c] for a rows x cols row-major matrix of esize-byte
 * elements (raw bits).  The tile is staged in shared memory; the variant
 * selects its layout.  The swizzled layouts are chosen per element size so
 * that both the row-wise fill and the column-wise drain are free of bank
 * conflicts ("CuTe Swizzle 学习手册", sections "冲突的典型场景" and
 * "不同矩阵配置的选择指南"; "CUDA 013 - Swizzle 的工作原理", sections
 * "如何避免 Bank Conflict", "swizzle 映射案例" and "行列位数"):
 *   esize 4 : 32 x 32 units, element Swizzle<5,0,5> (column XOR row);
 *   esize 8 : 16 x 16 units, element Swizzle<4,0,4>;
 *   esize 2 : 128-byte rows (64 elements) under the byte-address Swizzle<3,4,3>
 *             (16-byte chunk index XOR row mod 8; element Swizzle<3,3,3>),
 *             drained by 8 x 8 transposing matrix loads;
 *   esize 1 : 128 x 128-byte tiles under the byte-address Swizzle<3,4,7>
 *             (16-byte chunk index XOR (row / 16) mod 8), drained as 4 x 4
 *             byte blocks transposed in registers;
 *   esize 16 : 32 x 32 units, element Swizzle<5,0,5>.
 * SWZ_T_UNSWIZZLED uses the plain layout, SWZ_T_PADDED pads each row by one
 * element (by 16 bytes for esize 2); for esize 1 both run on 32 x 32 units.  SWZ_T_TMA is accepted for esize 2 only.
 *
 * dst: cols x rows elements; src: rows x cols elements; both device buffers.
 * rows, cols >= 0 (any value: edge tiles are handled element by element).
 *
 * Errors: SWZ_ERR_NULL, SWZ_ERR_PARAM (esize not in {1,2,4,8,16}, unknown
 * variant, SWZ_T_TMA with esize != 2), SWZ_ERR_SHAPE, SWZ_ERR_ALIGN,
 * SWZ_ERR_ALIAS, SWZ_ERR_CUDA.
 */
swz_status swz_transpose(void *dst, const void *src, int64_t rows, int64_t cols, int esize,
                         int variant, void *stream);

/*
 * Transpose fused with a forward relayout of its result.
 *
 * Sources: the transpose of swz_transpose, then the relayout of swz_relayout
 * ("CUDA 013 - Swizzle 的工作原理", sections "更通用的映射规则" and "使用示例");
 * the use is producing swizzled operand tiles directly, as in the
 * composition of Swizzle<3,4,3> with a (128, 64) row-major tile in "CuTe
 * Swizzle 学习手册", section "CuTe 中如何使用 Swizzle".
 *
 * Let T be the cols x rows transpose of src (rows x cols, row-major).  T is
 * cut into tiles of tile_elems consecutive elements and each tile is stored
 * in swizzled order: dst[t * tile_elems + sw(i)] = T[t * tile_elems + i].
 * One pass over HBM (the two steps apart would make two).  The staging is
 * SWZ_T_SWIZZLED's.
 *
 * rows, cols >= 0; tile_elems > 0 divides rows * cols and is a multiple of
 * 2^h (h as in swz_relayout: M + B, or M + |S| + B for S < 0); B, M, S as
 * in swz_relayout; esize 1, 2, 4, 8 or 16.  With S < 0 and M below the lane
 * bits of a 16-byte vector (2^M < 16 / esize) the transposed elements are
 * stored one by one (the swizzle then moves elements of one vector to
 * several), which is slower than the vector stores of every other case.
 * Errors: as swz_transpose, SWZ_ERR_PARAM for B, M, S, and SWZ_ERR_SHAPE
 * when tile_elems breaks the rules above.
 */
swz_status swz_transpose_relayout(void *dst, const void *src, int64_t rows, int64_t cols,
                                  int esize, int64_t tile_elems, int B, int M, int S,
                                  void *stream);

/*
 * Shared-memory bank-conflict profiler for warp access patterns.
 *
 * Model: 32 banks of 4 bytes, bank = (byte_addr / 4) % 32 ("CuTe Swizzle
 * 学习手册", section "Shared Memory 的 Bank 结构"); lanes touching different
 * 4-byte words of one bank are served one after another (N-way), lanes
 * touching the same word are served together, including two 16-bit halves
 * of one word ("CuTe Swizzle 学习手册", section "什么情况下产生冲突";
 * "CUDA 013 - Swizzle 的工作原理", section "什么是 Bank Conflict"; "NVIDIA CuTe
 * Swizzle").  An access wider than one pass can carry takes several passes
 * and that minimum is not a conflict ("NVIDIA CuTe Swizzle").  The split
 * into passes is not fixed by those sources; this library reads it as: up to
 * 4 bytes per lane, one pass of 32 lanes; 8 bytes, two passes (lanes 0-15,
 * 16-31); 16 bytes, four passes of 8 lanes.  In a pass each active lane
 * touches the words floor(a/4) .. floor((a + w - 1)/4); the pass costs the
 * largest number of distinct words in one bank.
 *
 * byte_addrs  : device, n x 32 uint32 byte addresses (pattern p, lane l at
 *               p * 32 + l).
 * active      : device, n uint32 lane masks, or NULL for all lanes active.
 * access_bytes: 1, 2, 4, 8 or 16.
 * ways        : device, n int32: the worst pass cost (1 = conflict-free,
 *               0 = no active lane).
 * wavefronts  : device, n int32: the sum of the pass costs.
 *
 * Errors: SWZ_ERR_NULL, SWZ_ERR_PARAM, SWZ_ERR_SHAPE (n < 0), SWZ_ERR_CUDA.
 */
swz_status swz_bank_profile(const uint32_t *byte_addrs, const uint32_t *active, int64_t n,
                            int access_bytes, int32_t *ways, int32_t *wavefronts,
                            void *stream);

/*
 * Shared-memory staging probe: a diagnostic for hardware bank-conflict
 * counters, not a data path.  A column read of a row-major shared tile puts
 * every lane in one bank ("CuTe Swizzle 学习手册", section "冲突的典型场景");
 * the transpose stagings avoid it by XOR-ing the column ("Swizzle 数学公式")
 * or padding the rows ("CUDA 013 - Swizzle 的工作原理", section "如何避免
 * Bank Conflict").  This call launches `ctas` CTAs that each fill and drain
 * one shared tile `iters` times with exactly the shared-memory instructions
 * and addresses of the swz_transpose staging of that element size and
 * variant (esize 4 / 8 / 2: SWZ_T_SWIZZLED, SWZ_T_UNSWIZZLED, SWZ_T_PADDED;
 * esize 2 also SWZ_T_TMA: the swizzled tile, whose transposing reads are
 * written with stmatrix into a second tile under the same swizzle, as the
 * TMA transpose does before its tensor store; esize 1: SWZ_T_SWIZZLED, the
 * 128 x 128-byte tile), on values held in registers.  The SWZ_T_TMA replay
 * fills the input tile with 16-byte stores where the transpose uses a tensor
 * load, so it shows the LSU side of that kernel without any tensor copy.
 *
 * gsrc, gdst, gbytes: optional device buffers of gbytes bytes (a multiple of
 * 16, 16-byte aligned, not overlapping).  NULL: the kernel makes no global
 * memory access at all.  Given: each iteration also streams one 16-byte load
 * from gsrc per fill vector and one 16-byte store to gdst per drain vector,
 * as the transpose does, cycling through the buffers.
 * sink: optional device array of `ctas` words; each CTA writes a checksum of
 * what it read after its last iteration (NULL: nothing is written).
 *
 * Errors: SWZ_ERR_PARAM (esize, variant), SWZ_ERR_SHAPE (iters, ctas < 0,
 * ctas >= 2^31, gbytes), SWZ_ERR_ALIGN, SWZ_ERR_ALIAS, SWZ_ERR_CUDA.
 */
swz_status swz_staging_probe(int esize, int variant, int iters, const void *gsrc, void *gdst,
                             int64_t gbytes, uint32_t *sink, int64_t ctas, void *stream);

/*
 * Slice collision ("cutlass 入门", section "swizzle 融入 layout 优化").
 *
 * A is the largest index of a slice, so its set bits are the bits that can
 * change.  C = A & ~sw(A).  C == 0 means no (Y_i, Z_i) pair of the swizzle has
 * both bits active, so on this slice the swizzle equals a plain layout and
 * can be folded into it; each set bit of C names a colliding Z bit.
 *
 * Host function, synchronous, no GPU involved.  C_out: host pointer.
 * Errors: SWZ_ERR_NULL (C_out NULL), SWZ_ERR_PARAM (B, M, S out of the range
 * of swz_relayout, or B + M + |S| > 64).
 */
swz_status swz_slice_collision(uint64_t A, int B, int M, int S, uint64_t *C_out);

/*
 * The plain layout that replaces the swizzle on a slice ("cutlass 入门",
 * section "swizzle 融入 layout 优化": when no (Y_i, Z_i) pair is active, the
 * swizzle composed with the slice equals a plain layout).
 *
 * If swz_slice_collision(A) is 0, writes for each set bit of A, from the
 * lowest, its stride strides[k] = sw(2^bit) and the count to *n_bits, so that
 * sw(x) = sum over the set bits of x of their strides, for every x whose bits
 * are a subset of A; returns SWZ_OK.  Otherwise writes nothing and returns
 * SWZ_ERR_UNSUPPORTED (the slice keeps a real XOR).  strides: host array of
 * at least 64 entries.  Host function, synchronous.
 * Errors: SWZ_ERR_NULL, SWZ_ERR_PARAM (as swz_slice_collision).
 */
swz_status swz_slice_layout(uint64_t A, int B, int M, int S, uint64_t *strides, int *n_bits);

/*
 * Batched slice collision on the GPU: C[k] = A[k] & ~sw(A[k]) for n masks.
 * A, C: device arrays of n uint64; C may be A itself (in place), otherwise
 * the two must not overlap (SWZ_ERR_ALIAS).  Same parameter rules as
 * swz_slice_collision; SWZ_ERR_SHAPE for n < 0 or n * 8 bytes overflowing.
 */
swz_status swz_slice_collision_batch(const uint64_t *A, int64_t n, int B, int M, int S,
                                     uint64_t *C, void *stream);

/*
 * Device status of bounded waits.
 *
 * The SWZ_T_TMA transpose waits on shared-memory barriers that its tensor
 * copies complete; every such wait gives up after a time limit (2 s), records
 * the expiry in a per-device status word and returns, leaving the context
 * usable.  This call synchronises `stream`, then reads and clears the status
 * word of the current device: SWZ_ERR_TIMEOUT if a wait gave up since the
 * last call, SWZ_OK otherwise, SWZ_ERR_CUDA if the synchronisation or the
 * read failed.  The status word is one 4-byte device allocation per device,
 * made by the first SWZ_T_TMA call on that device and kept until exit.
 */
swz_status swz_device_status(void *stream);

/*
 * Self-test of the bounded wait: launches the SWZ_T_TMA transpose kernel
 * with no tensor copy issued, so each of its waits expires after wait_ns
 * nanoseconds; the kernel records SWZ_ERR_TIMEOUT and returns without
 * writing dst.  Read the outcome with swz_device_status().  rows, cols > 0,
 * cols a multiple of 8, src 16-byte aligned (SWZ_ERR_SHAPE, SWZ_ERR_ALIGN).
 */
swz_status swz_selftest_tma_timeout(void *dst, const void *src, int64_t rows, int64_t cols,
                                    uint64_t wait_ns, void *stream);

/*
 * The SWZ_T_TMA transpose without any allocation by the library.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot let a library allocate device memory: a serving loop whose device
 * memory is planned ahead and owned by its own pool, a process whose device
 * memory is already fully reserved by another allocator, or code that must
 * not block on the allocator.  swz_transpose(..., SWZ_T_TMA) makes one
 * cudaMalloc (its 4-byte status word) on its first call on each device; this
 * entry point instead keeps that status word in a fixed 256-byte array in
 * the library's device data (every GPU that loads the library holds that
 * array until the process exits).  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Computes the same result as swz_transpose(dst, src, rows, cols, 2,
 * SWZ_T_TMA, stream): out[c][r] = in[r][c] for 16-bit elements (raw bits),
 * with the same kernel (one tile per CTA: a tensor load under the hardware
 * 128-byte swizzle, conflict-free transposing matrix reads, and a tensor
 * store when dst is 16-byte aligned and rows is a multiple of 8, element
 * stores otherwise); only the place of its status word differs.  Both fall
 * back to the shared-memory-staged swizzled kernel when src is not 16-byte
 * aligned or cols is not a multiple of 8.
 *
 * dst, src  : device buffers of rows x cols 2-byte elements (caller-owned).
 * rows, cols: 0 <= rows, cols < 2^31 (the TMA coordinate range); larger
 *             requests are refused with SWZ_ERR_SHAPE.  The call needs one
 *             4-byte status word of the array for any matrix size.
 * timed_out : optional host pointer.  NULL: the call returns once the work
 *             is enqueued, and a bounded wait that gives up goes unreported
 *             (dst is then incomplete; the next call clears the status
 *             word).  Non-NULL: the call waits for `stream`, stores 1 if one
 *             of the kernel's bounded waits gave up (dst is then incomplete
 *             and SWZ_ERR_TIMEOUT is returned), 0 otherwise.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, once per device, with that device current); make
 * that first call before any stream capture.  Every call shares the array:
 * each call clears the status word on `stream` before its kernel runs, and
 * calls whose work overlaps on the GPU (on different streams) race on it.
 *
 * Errors: SWZ_ERR_NULL, SWZ_ERR_SHAPE, SWZ_ERR_ALIGN (dst or src not 2-byte
 * aligned), SWZ_ERR_ALIAS, SWZ_ERR_CUDA, SWZ_ERR_TIMEOUT (timed_out only).
 */
swz_status swz_transpose_tma_noalloc(void *dst, const void *src, int64_t rows, int64_t cols,
                                     uint32_t *timed_out, void *stream);

/*
 * Self-test of swz_transpose_tma_noalloc's timeout report: the same call with
 * no tensor copy issued, so each bounded wait of its kernel gives up after
 * wait_ns nanoseconds and the kernel records the expiry in the fixed array's
 * status word and returns without writing dst.  Waits for `stream`; stores 1
 * in *timed_out and returns SWZ_ERR_TIMEOUT when the expiry was reported.
 * rows, cols > 0, cols a multiple of 8, src 16-byte aligned (SWZ_ERR_SHAPE,
 * SWZ_ERR_ALIGN); timed_out must not be NULL (SWZ_ERR_NULL).  Allocates
 * nothing.  Host function that launches one kernel.
 */
swz_status swz_selftest_noalloc_timeout(void *dst, const void *src, int64_t rows, int64_t cols,
                                        uint64_t wait_ns, uint32_t *timed_out, void *stream);

/*
 * Text map of a swizzled tile, the counterpart of CuTe's print_layout
 * ("CuTe Swizzle 学习手册", section "如何验证 Swizzle 是否正确消除冲突": print
 * each element's swizzled offset and its bank; with no bank repeated within
 * a 128-byte row segment the layout is conflict-free for row access).
 *
 * One line per tile row; for each column "physical_offset/bank", separated
 * by single spaces, where physical_offset = sw(r * cols + c) and bank =
 * (physical_offset * esize / 4) % 32.  Writes at most cap bytes including
 * the terminating NUL into buf (buf may be NULL when cap is 0) and returns
 * the length of the whole text, excluding the NUL, or -1 for bad arguments
 * (rows, cols < 0, esize < 1, B, M, S out of range).  Host function.
 */
int64_t swz_layout_text(char *buf, int64_t cap, int64_t rows, int64_t cols, int esize, int B, int M,
                        int S);

/* sw(x) on the host (the same function the kernels apply). */
uint64_t swz_apply(uint64_t x, int B, int M, int S);

/* A static, human-readable name of a status code. */
const char *swz_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int swz_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SWZ_H */
