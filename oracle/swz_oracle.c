/*
 * swz_oracle.c -- plain, slow CPU oracle for the XOR-swizzle data-movement path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA library; it is written from the pages' definitions
 * with one element per loop iteration and no blocking or reordering.
 *
 * Sources (page title, section):
 *   [P1] "NVIDIA CuTe Swizzle" -- the bit diagram, sub-word broadcast,
 *        "minimum steps are not a conflict".
 *   [P2] "CuTe Swizzle 学习手册" -- bank structure, conflict rules,
 *        "Swizzle 数学公式".
 *   [P3] "cutlass 入门" -- "swizzle 融入 layout 优化" (slice collision).
 *   [P4] "CUDA 013 - Swizzle 的工作原理" -- "CuTe 通用 swizzle 映射规则解析"
 *        (the Z and Y fields, AA = ZZ xor YY), "计算公式" (the names base,
 *        bits, shift), "更通用的映射规则" (offset-based rule, worked
 *        example), "什么是 Bank Conflict".
 *
 * Parity status per function (what pins it is listed in the test suite):
 *   orc_swizzle            pinned (worked example, 2-D closed forms, bit diagrams);
 *                          negative shifts pinned to the positive ones by the
 *                          bit-reversal mirror identity (the reading of the
 *                          negative case itself is argued, not printed)
 *   orc_relayout           pinned (reduces to orc_swizzle + byte copies)
 *   orc_transpose          pinned (textbook transpose, explicit small cases)
 *   orc_transpose_relayout the two pinned steps above, in that order
 *   orc_bank_profile       pinned for every access width: 1, 2, 4 by the
 *                          pages' bank rules; 16 by the ldmatrix.m8n8.x4
 *                          note of [P1] (four reads, one per 8 x 8 matrix);
 *                          8 by [P1]'s 128-byte operation size (its grouping
 *                          into consecutive half-warps is a reading).
 *   orc_slice_collision    pinned (truth tables, brute-force additivity)
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <stdio.h>

/* Status codes of this oracle (independent of the library's codes). */
#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_NOT_CLOSED 2

/* Bit p of v (0 beyond the 64 bits of an offset). */
static int orc_bit(uint64_t v, int p)
{
    if (p < 0 || p >= 64)
        return 0;
    return (int)((v >> p) & 1u);
}

/*
 * The swizzle of one offset, bit by bit, as [P1]'s bit diagram and
 * [P4] "CuTe 通用 swizzle 映射规则解析" define it: the lowest `base` bits
 * take no part; a field Z of `bits` bits starts at bit `base`, a field Y of
 * the same width starts `shift` bits above it; in the result, bit i of Z
 * becomes (bit i of Z) xor (bit i of Y), and every bit outside Z is the
 * input's.  The output is built one bit at a time from the input, so no
 * written bit feeds a later read.
 *
 * Negative shift.  [P1]'s bit-diagram comment makes SShift the distance the
 * YYY mask is moved to land on ZZZ, rightward when positive and leftward when
 * negative, and keeps the lowest MBase bits constant.  So for a negative
 * shift YYY is the lower of the two fields, and both fields stay above the
 * `base` constant bits: Y starts at bit `base` and Z starts -shift bits
 * above it.  (The pages print no example of a negative shift; this is the
 * reading that keeps the lowest `base` bits out of the map, as for a
 * positive shift.)
 */
uint64_t orc_swizzle(uint64_t offset, int base, int bits, int shift)
{
    uint64_t out = offset;
    int zlo = shift >= 0 ? base : base - shift;   /* the field that is written */
    int ylo = shift >= 0 ? base + shift : base;   /* the field that is read */
    int i;
    for (i = 0; i < bits; ++i) {
        int zpos = zlo + i;
        int ypos = ylo + i;
        int v;
        if (zpos >= 64)
            break;
        v = orc_bit(offset, zpos) ^ orc_bit(offset, ypos);
        if (v)
            out |= (uint64_t)1 << zpos;
        else
            out &= ~((uint64_t)1 << zpos);
    }
    return out;
}

/*
 * Batched relayout.  [P4] "使用示例" example 1: the element at logical offset
 * `o` of a tile is accessed at the swizzled offset swizzle(o).  Forward
 * (direction 0) stores logical element i at physical position swizzle(i);
 * inverse (direction 1) reads the physical position swizzle(i) back into
 * logical position i.  Offsets are local to each tile of tile_elems elements.
 */
int orc_relayout(void *dst, const void *src, int64_t n_tiles, int64_t tile_elems,
                 int esize, int base, int bits, int shift, int direction)
{
    unsigned char *d = (unsigned char *)dst;
    const unsigned char *s = (const unsigned char *)src;
    int64_t t, i;
    if (!dst || !src || n_tiles < 0 || tile_elems < 0 || esize <= 0)
        return ORC_BAD_ARG;
    if (direction != 0 && direction != 1)
        return ORC_BAD_ARG;
    for (t = 0; t < n_tiles; ++t) {
        int64_t tile0 = t * tile_elems;
        for (i = 0; i < tile_elems; ++i) {
            uint64_t j = orc_swizzle((uint64_t)i, base, bits, shift);
            if (j >= (uint64_t)tile_elems)
                return ORC_NOT_CLOSED;
            if (direction == 0)
                memcpy(d + (size_t)(tile0 + (int64_t)j) * esize,
                       s + (size_t)(tile0 + i) * esize, (size_t)esize);
            else
                memcpy(d + (size_t)(tile0 + i) * esize,
                       s + (size_t)(tile0 + (int64_t)j) * esize, (size_t)esize);
        }
    }
    return ORC_OK;
}

/*
 * Relayout of selected logical offsets only: for each global logical index
 * idx[k] (tile * tile_elems + local), out_pos[k] receives the global physical
 * index that element lands on (direction 0), or the global physical index it
 * is read from (direction 1).  Used to check samples of very large buffers.
 */
int orc_relayout_positions(const int64_t *idx, int64_t n, int64_t tile_elems,
                           int base, int bits, int shift, int64_t *out_pos)
{
    int64_t k;
    if (!idx || !out_pos || tile_elems <= 0)
        return ORC_BAD_ARG;
    for (k = 0; k < n; ++k) {
        int64_t tile = idx[k] / tile_elems;
        int64_t local = idx[k] % tile_elems;
        uint64_t j = orc_swizzle((uint64_t)local, base, bits, shift);
        if (j >= (uint64_t)tile_elems)
            return ORC_NOT_CLOSED;
        out_pos[k] = tile * tile_elems + (int64_t)j;
    }
    return ORC_OK;
}

/* Matrix transpose, the textbook definition: out[c][r] = in[r][c]. */
int orc_transpose(void *dst, const void *src, int64_t rows, int64_t cols, int esize)
{
    unsigned char *d = (unsigned char *)dst;
    const unsigned char *s = (const unsigned char *)src;
    int64_t r, c;
    if (!dst || !src || rows < 0 || cols < 0 || esize <= 0)
        return ORC_BAD_ARG;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c)
            memcpy(d + (size_t)(c * rows + r) * esize,
                   s + (size_t)(r * cols + c) * esize, (size_t)esize);
    return ORC_OK;
}

/*
 * Transpose, then forward relayout of the transposed matrix: the cols x rows
 * result is cut into tiles of tile_elems consecutive elements and each tile is
 * stored in swizzled order.  The two steps in that order, through a scratch
 * copy of the transposed matrix (tmp, rows * cols elements, caller-owned).
 */
int orc_transpose_relayout(void *dst, const void *src, void *tmp, int64_t rows, int64_t cols, int esize,
                           int64_t tile_elems, int base, int bits, int shift)
{
    int rc;
    if (tile_elems <= 0 || (rows * cols) % tile_elems != 0)
        return ORC_BAD_ARG;
    rc = orc_transpose(tmp, src, rows, cols, esize);
    if (rc != ORC_OK)
        return rc;
    return orc_relayout(dst, tmp, (rows * cols) / tile_elems, tile_elems, esize, base, bits, shift, 0);
}

/*
 * Bank model for one warp-wide shared-memory access.
 *
 * [P2] "Shared Memory 的 Bank 结构": 32 banks of 4 bytes, bank =
 *   (byte_addr / 4) % 32.
 * [P2] "什么情况下产生冲突" / [P4] "什么是 Bank Conflict": threads that touch
 *   different addresses in the same bank are served one after the other;
 *   N distinct addresses in one bank make an N-way conflict.  Threads that
 *   touch the same address are served together (broadcast).
 * [P1]: two 16-bit values in one 32-bit word are broadcast together, so the
 *   unit of "same address" is the 4-byte word.
 * [P1]: an operation that moves more data than one pass can carry needs
 *   several passes; that minimum is not a conflict.  Conflicts are counted
 *   within each pass.
 *
 * [P1], the ldmatrix.m8n8.x4 note: a 16 x 16 fp16 block (512 bytes) is read
 *   in four warp reads, one per 8 x 8 matrix; matrix m's row addresses come
 *   from lanes 8m .. 8m+7 (PTX ISA), so w = 16 is four passes of 8 lanes.
 * [P1]: one operation serves at most 64 fp16 values (128 bytes), so w = 8 is
 *   two passes of 16 lanes; taking them as lanes 0-15 and 16-31 is the
 *   reading (the pages do not name the lanes).  w <= 4 is one pass over all
 *   32 lanes.  In each pass
 * every active lane touches the words floor(a/4) .. floor((a+w-1)/4); the
 * pass costs the largest number of distinct words that fall in one bank.
 * ways = largest pass cost, wavefronts = sum of pass costs.
 *
 * addrs: n patterns of 32 byte addresses; active: n lane masks or NULL (all
 * lanes active).  Outputs ways[n], wavefronts[n].
 */
int orc_bank_profile(const uint32_t *addrs, const uint32_t *active, int64_t n,
                     int width, int32_t *ways, int32_t *wavefronts)
{
    int64_t p;
    int passes, lanes_per_pass;
    if (!addrs || !ways || !wavefronts || n < 0)
        return ORC_BAD_ARG;
    if (width != 1 && width != 2 && width != 4 && width != 8 && width != 16)
        return ORC_BAD_ARG;
    passes = (width <= 4) ? 1 : width / 4;
    lanes_per_pass = 32 / passes;
    for (p = 0; p < n; ++p) {
        uint32_t mask = active ? active[p] : 0xffffffffu;
        int32_t worst = 0, total = 0;
        int pass;
        for (pass = 0; pass < passes; ++pass) {
            /* distinct words touched in this pass; at most 8 lanes x 5 words
               or 32 lanes x 2 words */
            uint64_t words[64];
            int n_words = 0, lane, k, bank, cost = 0;
            for (lane = pass * lanes_per_pass; lane < (pass + 1) * lanes_per_pass; ++lane) {
                uint64_t a, first, last, wd;
                if (!((mask >> lane) & 1u))
                    continue;
                a = addrs[p * 32 + lane];
                first = a / 4;
                last = (a + (uint64_t)width - 1) / 4;
                for (wd = first; wd <= last; ++wd) {
                    int seen = 0;
                    for (k = 0; k < n_words; ++k)
                        if (words[k] == wd)
                            seen = 1;
                    if (!seen)
                        words[n_words++] = wd;
                }
            }
            for (bank = 0; bank < 32; ++bank) {
                int count = 0;
                for (k = 0; k < n_words; ++k)
                    if ((int)(words[k] % 32) == bank)
                        ++count;
                if (count > cost)
                    cost = count;
            }
            if (cost > worst)
                worst = cost;
            total += cost;
        }
        ways[p] = worst;
        wavefronts[p] = total;
    }
    return ORC_OK;
}

/*
 * [P3] "swizzle 融入 layout 优化": A is the slice's largest index (its bits
 * are the bits that can change).  collision = A & ~swizzle(A); a set bit
 * marks a pair of fields whose y bit and z bit are both active, in which case
 * the swizzle cannot be folded into a plain layout.
 */
uint64_t orc_slice_collision(uint64_t A, int base, int bits, int shift)
{
    return A & ~orc_swizzle(A, base, bits, shift);
}

/*
 * Brute-force check of the property the collision rule predicts: the
 * swizzle, restricted to every x whose bits are a subset of A, equals a plain
 * layout sum_i x_i * swizzle(2^i) (integer sum of per-bit strides).
 * Returns 1 when it does, 0 when some subset breaks it.
 */
int orc_slice_is_layout(uint64_t A, int base, int bits, int shift)
{
    uint64_t x = 0;
    for (;;) {
        uint64_t sum = 0;
        int i;
        for (i = 0; i < 64; ++i)
            if ((x >> i) & 1u)
                sum += orc_swizzle((uint64_t)1 << i, base, bits, shift);
        if (sum != orc_swizzle(x, base, bits, shift))
            return 0;
        if (x == A)
            break;
        x = (x - A) & A; /* next subset of A in increasing order */
    }
    return 1;
}

/*
 * Text dump of a swizzled rows x cols tile ([P2] "如何验证 Swizzle 是否正确消除
 * 冲突": print the mapping and the bank of each element).  One line per row:
 * for every column "physical_offset/bank".  Returns the number of characters
 * needed (excluding the terminator); writes at most cap bytes.
 */
int64_t orc_dump_layout(char *buf, int64_t cap, int64_t rows, int64_t cols, int esize,
                        int base, int bits, int shift)
{
    int64_t r, c, used = 0;
    char tmp[64];
    for (r = 0; r < rows; ++r) {
        for (c = 0; c < cols; ++c) {
            uint64_t phys = orc_swizzle((uint64_t)(r * cols + c), base, bits, shift);
            uint64_t bank = (phys * (uint64_t)esize / 4) % 32;
            int len = snprintf(tmp, sizeof tmp, "%s%llu/%llu", c ? " " : "",
                               (unsigned long long)phys, (unsigned long long)bank);
            if (buf && used + len < cap)
                memcpy(buf + used, tmp, (size_t)len);
            used += len;
        }
        if (buf && used + 1 < cap)
            buf[used] = '\n';
        used += 1;
    }
    if (buf && cap > 0)
        buf[used < cap ? used : cap - 1] = '\0';
    return used;
}
