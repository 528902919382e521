"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages print (fixtures under tests/golden/, each citing its page and section),
a coordinate-level restatement of a 2-D mapping the pages describe, the bit
diagrams read position by position, closed forms and invariants, and brute
force on tiny inputs.
"""
import itertools

import numpy as np
import pytest

from conftest import read_golden

SWEEP = [(B, M, S) for B in range(1, 6) for M in range(0, 5) for S in range(B, 8)]
CONFIG_SWIZZLES = [(3, 3, 3), (3, 4, 3), (5, 2, 5), (5, 0, 5), (4, 0, 4)]


# ---------------------------------------------------------------- swizzle ---

def test_worked_example_673(orc):
    g = {row[0]: row[1] for row in read_golden("worked_example_673.txt")}
    rows, cols = int(g["rows"]), int(g["cols"])
    base, bits, shift = int(g["base"]), int(g["bits"]), int(g["shift"])
    r, c = int(g["logical_row"]), int(g["logical_col"])
    off = r * cols + c
    assert off == int(g["offset"]) == int(g["offset_binary"], 2)
    sw = orc.swizzle(off, B=bits, M=base, S=shift)
    assert sw == int(g["swizzled"]) == int(g["swizzled_binary"], 2)
    assert divmod(sw, cols) == (int(g["physical_row"]), int(g["physical_col"]))
    # the same fact through the relayout: the element with logical value 673
    # of an int[32][64] array lands at physical position 683
    iota = np.arange(rows * cols, dtype=np.int32)
    phys = orc.relayout(iota, tile_elems=rows * cols, B=bits, M=base, S=shift, direction=0)
    assert phys.reshape(rows, cols)[int(g["physical_row"]), int(g["physical_col"])] == off


def _mapping_32x32(y, x):
    # 32 x 32 words: the column index is XOR-ed with the row index
    return y, x ^ y


def _mapping_64x32(y, x):
    # 64 rows: the two 32-row halves are swizzled the same way (row taken mod 32)
    return y, x ^ (y & 31)


def _mapping_32x64(y, x):
    # 64 columns: each 32-column half is swizzled on its own
    half, within = divmod(x, 32)
    return y, half * 32 + (within ^ y)


def _mapping_half_pairs(y, x):
    # 16-bit data, two neighbours kept together: swizzle the pair index
    pair, lane = divmod(x, 2)
    return y, (pair ^ y) * 2 + lane


@pytest.mark.parametrize("rows,cols,mapping,params", [
    (32, 32, _mapping_32x32, (5, 0, 5)),
    (64, 32, _mapping_64x32, (5, 0, 5)),
    (32, 64, _mapping_32x64, (5, 0, 6)),
    (32, 64, _mapping_half_pairs, (5, 1, 5)),
])
def test_two_d_mappings(orc, rows, cols, mapping, params):
    """"CUDA 013 - Swizzle 的工作原理", section "swizzle 映射案例": the four 2-D
    mappings equal the offset rule of section "计算公式" with these parameters."""
    B, M, S = params
    for y in range(rows):
        for x in range(cols):
            py, px = mapping(y, x)
            assert orc.swizzle(y * cols + x, B=B, M=M, S=S) == py * cols + px


def _diagram_positions(pattern_or_tokens):
    """Return (z_positions, y_positions), least significant first."""
    if isinstance(pattern_or_tokens, str):
        tokens = list(pattern_or_tokens)
    else:
        tokens = pattern_or_tokens
    assert len(tokens) == 32
    z, y = {}, {}
    for i, t in enumerate(tokens):
        bit = 31 - i
        if t.startswith("Z"):
            z[bit] = t
        elif t.startswith("Y"):
            y[bit] = t
    zs, ys = sorted(z), sorted(y)
    return zs, ys


def test_bit_diagrams(orc):
    """"NVIDIA CuTe Swizzle" (diagram and example) and "cutlass 入门"
    (section "具体过程"): read the field positions off each diagram and check the
    oracle bit by bit: each Z bit becomes Z xor the Y bit in the same place of
    its field, every other bit is kept."""
    rows = {r[0]: r[1:] for r in read_golden("bit_diagrams.txt")}
    expected_params = {}
    rng = np.random.default_rng(12345)
    for name, fields in rows.items():
        pattern = fields[0] if len(fields) == 1 else fields
        zs, ys = _diagram_positions(pattern)
        assert len(zs) == len(ys) > 0
        assert zs == list(range(zs[0], zs[0] + len(zs)))
        assert ys == list(range(ys[0], ys[0] + len(ys)))
        # MBase is where the lower field starts; SShift is Y's distance from Z
        # (negative when Y is the lower field)
        B, M, S = len(zs), min(zs[0], ys[0]), ys[0] - zs[0]
        expected_params[name] = (B, M, S)
        for x in itertools.chain(rng.integers(0, 2**32, 2000, dtype=np.uint64).tolist(),
                                 [0, 2**32 - 1]):
            want = 0
            for bit in range(32):
                v = (x >> bit) & 1
                if bit in zs:
                    v ^= (x >> ys[zs.index(bit)]) & 1
                want |= v << bit
            assert orc.swizzle(int(x), B=B, M=M, S=S) == want
    # counting the characters gives these parameters
    assert expected_params == {"p1_diagram": (3, 4, 10), "p1_example": (2, 3, 11),
                               "p3_tokens": (4, 4, 11), "p1_diagram_negative_shift": (3, 4, -10)}


@pytest.mark.parametrize("B,M,S", SWEEP + CONFIG_SWIZZLES)
def test_swizzle_invariants(orc, B, M, S):
    """Consequences of the definition, exhaustively over offsets 0..65535."""
    x = np.arange(1 << 16, dtype=np.uint64)
    sw = np.array([orc.swizzle(int(v), B=B, M=M, S=S) for v in x], dtype=np.uint64)
    # a bijection of 0..65535 onto itself
    assert np.array_equal(np.sort(sw), x)
    # self-inverse when the two fields do not overlap (S >= B)
    if S >= B:
        back = np.array([orc.swizzle(int(v), B=B, M=M, S=S) for v in sw], dtype=np.uint64)
        assert np.array_equal(back, x)
    # the low M bits are kept: groups of 2^M elements stay contiguous and in order
    low = (1 << M) - 1
    assert np.array_equal(sw & np.uint64(low), x & np.uint64(low))
    # bits at and above M+B are only read, never written
    assert np.array_equal(sw >> np.uint64(M + B), x >> np.uint64(M + B))


NEGATIVE = [(B, M, -s) for B in range(1, 6) for M in range(0, 5) for s in range(1, 8)]


def _bit_reverse(x: int, width: int) -> int:
    return int(format(x, f"0{width}b")[::-1], 2)


@pytest.mark.parametrize("B,M,s,Mr", [(3, 4, 10, 4), (2, 3, 11, 0), (1, 0, 1, 0), (3, 0, 1, 2),
                                      (3, 0, 3, 0), (5, 2, 5, 1), (4, 1, 2, 3), (2, 2, 7, 5)])
def test_negative_shift_mirrors_positive(orc, B, M, s, Mr):
    """A negative shift is the positive one seen in a mirror.  Reverse the bit
    order of a W-bit offset: the written field of Sw<B, M, s> (bits M .. M+B-1)
    lands on bits Mr+s .. Mr+s+B-1 and its read field (bits M+s ..) on
    Mr .. Mr+B-1, with W = M + Mr + s + B, and the pairing of the bits is kept.
    So Sw<B, Mr, -s> = reverse . Sw<B, M, s> . reverse on every W-bit offset:
    the positive swizzle, pinned by the pages' examples, fixes the negative
    one (YYY at MBase, ZZZ |SShift| above it, "NVIDIA CuTe Swizzle")."""
    W = M + Mr + s + B
    for x in range(1 << W) if W <= 14 else np.random.default_rng(W).integers(0, 1 << W, 20000).tolist():
        pos = orc.swizzle(_bit_reverse(int(x), W), B=B, M=M, S=s)
        assert orc.swizzle(int(x), B=B, M=Mr, S=-s) == _bit_reverse(pos, W)


@pytest.mark.parametrize("B,M,S", NEGATIVE)
def test_negative_shift_invariants(orc, B, M, S):
    """Negative shifts over offsets 0..65535: a bijection; its own inverse
    when the fields do not overlap (|S| >= B); the low M bits (and groups of
    2^M elements) kept; only the field |S| bits above MBase is written."""
    x = np.arange(1 << 16, dtype=np.uint64)
    sw = np.array([orc.swizzle(int(v), B=B, M=M, S=S) for v in x], dtype=np.uint64)
    assert np.array_equal(np.sort(sw), x)
    if -S >= B:
        back = np.array([orc.swizzle(int(v), B=B, M=M, S=S) for v in sw], dtype=np.uint64)
        assert np.array_equal(back, x)
    zlo = M - S
    keep = ~np.uint64(((1 << B) - 1) << zlo)
    assert np.array_equal(sw & keep, x & keep)
    assert np.array_equal(sw & np.uint64((1 << M) - 1), x & np.uint64((1 << M) - 1))


def test_swizzle_degenerate(orc):
    x = list(range(4096))
    # B = 0: the identity
    assert [orc.swizzle(v, B=0, M=3, S=3) for v in x] == x
    # S = 0: the field is XOR-ed with itself, so it is cleared; not a bijection
    vals = {orc.swizzle(v, B=3, M=2, S=0) for v in x}
    assert len(vals) < len(x)
    assert all(((orc.swizzle(v, B=3, M=2, S=0) >> 2) & 7) == 0 for v in x)
    # 1 <= S < B: still a bijection, but not always an involution
    sw = [orc.swizzle(v, B=3, M=0, S=1) for v in x]
    assert sorted(sw) == x
    assert any(orc.swizzle(s, B=3, M=0, S=1) != v for v, s in zip(x, sw))


# --------------------------------------------------------------- relayout ---

def test_relayout_roundtrip_and_closed(orc):
    rng = np.random.default_rng(0)
    for (B, M, S), esize in itertools.product([(3, 3, 3), (3, 0, 1), (2, 1, 1), (5, 2, 5)],
                                              [1, 2, 4, 8, 16]):
        tile = 1 << (B + M + S)
        dt = np.dtype(f"V{esize}")
        src = rng.integers(0, 256, 3 * tile * esize, dtype=np.uint8).view(dt)
        fwd = orc.relayout(src, tile_elems=tile, B=B, M=M, S=S, direction=0)
        inv = orc.relayout(fwd, tile_elems=tile, B=B, M=M, S=S, direction=1)
        assert inv.tobytes() == src.tobytes()
        if S >= B:
            inv2 = orc.relayout(fwd, tile_elems=tile, B=B, M=M, S=S, direction=0)
            assert inv2.tobytes() == src.tobytes()


@pytest.mark.parametrize("tile", [64, 48, 24])
def test_relayout_tile_local(orc, tile):
    """Tiles relayout independently: each tile of the batch equals a one-tile
    relayout of its own data.  48 and 24 are multiples of 2^(M+B) = 8 but not
    of the 64-element period of Swizzle<2,1,3>, so offsets taken over the
    whole batch instead of the tile would differ."""
    B, M, S = 2, 1, 3
    src = np.arange(3 * tile, dtype=np.int32)
    for direction in (0, 1):
        out = orc.relayout(src, tile_elems=tile, B=B, M=M, S=S, direction=direction)
        for t in range(3):
            alone = orc.relayout(np.ascontiguousarray(src[t * tile:(t + 1) * tile]), tile_elems=tile,
                                 B=B, M=M, S=S, direction=direction)
            assert np.array_equal(out[t * tile:(t + 1) * tile], alone)


def test_relayout_not_closed(orc):
    # a tile of 6 elements is not closed under Swizzle<2,0,1>: offset 4 maps to 6
    assert orc.swizzle(4, B=2, M=0, S=1) == 6
    with pytest.raises(ValueError):
        orc.relayout(np.arange(6, dtype=np.int32), tile_elems=6, B=2, M=0, S=1, direction=0)


def test_relayout_usage_loop(orc):
    """"CUDA 013 - Swizzle 的工作原理", section "使用示例", example 1: the element
    at logical (y, x) of int num[32][128] is accessed at the coordinate given by
    the swizzled offset split into row and column."""
    rows, cols, B, M, S = 32, 128, 5, 0, 7
    logical = np.arange(rows * cols, dtype=np.int32).reshape(rows, cols)
    phys = orc.relayout(logical.ravel(), tile_elems=rows * cols, B=B, M=M, S=S, direction=0)
    phys = phys.reshape(rows, cols)
    for y in range(rows):
        for x in range(cols):
            # 32 x 32 blocks: column bits 0..4 XOR row bits 0..4
            new_y, new_x = y, (x & ~31) | ((x & 31) ^ (y & 31))
            assert phys[new_y, new_x] == logical[y, x]


def test_relayout_positions(orc):
    idx = np.array([0, 673, 2047, 2048 + 673], dtype=np.int64)
    pos = orc.relayout_positions(idx, tile_elems=2048, B=5, M=0, S=6)
    assert pos.tolist() == [0, 683, orc.swizzle(2047, B=5, M=0, S=6), 2048 + 683]


# -------------------------------------------------------------- transpose ---

def test_transpose_small(orc):
    a = np.array([[1, 2, 3], [4, 5, 6]], dtype=np.int32)
    assert orc.transpose(a).tolist() == [[1, 4], [2, 5], [3, 6]]


@pytest.mark.parametrize("dtype", [np.uint8, np.uint16, np.float32, np.float64])
def test_transpose_matches_library(orc, dtype):
    rng = np.random.default_rng(7)
    a = rng.integers(0, 255, size=(37, 53)).astype(dtype)
    t = orc.transpose(a)
    assert np.array_equal(t, a.T)
    assert np.array_equal(orc.transpose(t), a)


def test_transpose_relayout_composes(orc):
    """The fused operation is the transpose followed by the forward relayout
    of the transposed matrix in tiles of tile_elems elements."""
    rng = np.random.default_rng(3)
    a = rng.integers(0, 2**16, size=(24, 40)).astype(np.uint16)
    got = orc.transpose_relayout(a, tile_elems=8 * 24, B=3, M=0, S=3)
    t = orc.transpose(a).ravel()
    assert np.array_equal(got, orc.relayout(t, tile_elems=8 * 24, B=3, M=0, S=3, direction=0))
    # the untouched case: B = 0 is the plain transpose
    assert np.array_equal(orc.transpose_relayout(a, tile_elems=24, B=0, M=0, S=3), a.T.ravel())
    # element (r, c) of the input lands in tile (c*rows + r) // te at sw(offset within the tile)
    te = 8 * 24
    for r, c in [(0, 0), (5, 7), (23, 39), (11, 20)]:
        off = c * 24 + r
        tile, loc = divmod(off, te)
        assert got[tile * te + orc.swizzle(loc, B=3, M=0, S=3)] == a[r, c]
    # a swizzle that is not its own inverse (S < B): the forward relayout puts
    # every element at sw(offset), which the inverse would not
    got1 = orc.transpose_relayout(a, tile_elems=te, B=3, M=0, S=1)
    for r in range(24):
        for c in range(40):
            tile, loc = divmod(c * 24 + r, te)
            assert got1[tile * te + orc.swizzle(loc, B=3, M=0, S=1)] == a[r, c]


# ------------------------------------------------------------- bank model ---

def _ways(orc, addrs, width, active=None):
    a = np.zeros(32, dtype=np.uint32)
    a[:len(addrs)] = addrs
    act = None
    if active is None and len(addrs) < 32:
        active = (1 << len(addrs)) - 1
    if active is not None:
        act = np.array([active], dtype=np.uint32)
    w, wf = orc.bank_profile(a.reshape(1, 32), width, act)
    return int(w[0]), int(wf[0])


def test_bank_column_fp32(orc):
    """"CuTe Swizzle 学习手册", section "冲突的典型场景": an 8 x 32 fp32 array read
    down column 0 puts every lane on bank 0; a row read is conflict-free."""
    col = [4 * (r * 32 + 0) for r in range(8)]
    assert _ways(orc, col, 4) == (8, 8)
    col32 = [4 * (r * 32 + 5) for r in range(32)]
    assert _ways(orc, col32, 4) == (32, 32)
    row = [4 * (0 * 32 + c) for c in range(32)]
    assert _ways(orc, row, 4) == (1, 1)


def test_bank_padding_and_xor(orc):
    """"CUDA 013 - Swizzle 的工作原理": a [32][33] array and the (y, x ^ y)
    mapping both make a column read conflict-free."""
    padded = [4 * (r * 33 + 7) for r in range(32)]
    assert _ways(orc, padded, 4) == (1, 1)
    xor = [4 * (r * 32 + (7 ^ r)) for r in range(32)]
    assert _ways(orc, xor, 4) == (1, 1)
    for x in range(32):
        sw = [4 * orc.swizzle(r * 32 + x, B=5, M=0, S=5) for r in range(32)]
        assert _ways(orc, sw, 4) == (1, 1)


def test_bank_fp16_64_columns(orc):
    """"CuTe Swizzle 学习手册": an 8 x 64 fp16 array (128-byte rows) read down a
    column.  Unswizzled: 8-way.  Swizzle<3,3,3> in element units: conflict
    free, both as 2-byte scalars and as 16-byte row vectors.  Element-unit
    Swizzle<3,4,3> on the same rows is 2-way (the "matrix too narrow" case of
    the pitfalls table)."""
    for col in range(64):
        plain = [2 * (r * 64 + col) for r in range(8)]
        assert _ways(orc, plain, 2)[0] == 8
        s333 = [2 * orc.swizzle(r * 64 + col, B=3, M=3, S=3) for r in range(8)]
        assert _ways(orc, s333, 2) == (1, 1)
    for chunk in range(8):
        vec333 = [2 * orc.swizzle(r * 64 + 8 * chunk, B=3, M=3, S=3) for r in range(8)]
        assert _ways(orc, vec333, 16) == (1, 1)
        vec_plain = [2 * (r * 64 + 8 * chunk) for r in range(8)]
        assert _ways(orc, vec_plain, 16) == (8, 8)
        s343 = [2 * orc.swizzle(r * 64 + 8 * chunk, B=3, M=4, S=3) for r in range(8)]
        assert _ways(orc, s343, 2)[0] == 2


def test_bank_usage_examples(orc):
    """"CUDA 013 - Swizzle 的工作原理", section "使用示例": with each example's
    parameters, reading one column of basic elements down the rows is
    conflict-free within every pass."""
    for name, esize, rows, cols, base, bits, shift in read_golden("usage_examples.txt"):
        esize, rows, cols = int(esize), int(rows), int(cols)
        base, bits, shift = int(base), int(bits), int(shift)
        unit = esize << base                      # bytes kept together
        lanes = 32 if unit <= 4 else 32 // (unit // 4)
        per_row = cols >> base                    # basic elements per row
        for col_unit in range(per_row):
            addrs = []
            for r in range(min(rows, lanes)):
                off = r * cols + (col_unit << base)
                addrs.append(esize * orc.swizzle(off, B=bits, M=base, S=shift))
            w, _ = _ways(orc, addrs, unit)
            assert w == 1, (name, col_unit)


def test_bank_broadcast(orc):
    """Same word: broadcast ("CuTe Swizzle 学习手册"); two 16-bit halves of one
    word are served together ("NVIDIA CuTe Swizzle")."""
    assert _ways(orc, [128] * 32, 4) == (1, 1)
    assert _ways(orc, [0, 2] * 16, 2) == (1, 1)
    assert _ways(orc, [0, 1, 2, 3] * 8, 1) == (1, 1)


def test_bank_minimum_passes(orc):
    """"NVIDIA CuTe Swizzle": a 16 x 16 fp16 tile (256 elements, 512 bytes) read
    by one warp takes four passes; that is the minimum, not a conflict."""
    addrs = [16 * l for l in range(32)]
    ways, wavefronts = _ways(orc, addrs, 16)
    assert ways == 1 and wavefronts == 4


def test_bank_ldmatrix_x4_passes(orc):
    """"NVIDIA CuTe Swizzle", the note on ldmatrix.m8n8.x4: the 16 x 16 fp16
    block (512 bytes) is four warp reads, one per 8 x 8 matrix, and only a
    conflict inside one of them counts.  ldmatrix .x4 takes matrix m's eight
    row addresses from lanes 8m .. 8m+7 (PTX ISA, ldmatrix).  In the page's
    (-1, 64) fp16 layout under Swizzle<3,3,3>, lanes i and 8 + i hit the same
    banks (rows i and 8 + i share a chunk position) but sit in different
    matrices: no conflict, four passes.  Unswizzled, each matrix's eight rows
    share one chunk position: 8-way in every pass."""
    for r0, c0 in [(0, 0), (16, 8), (40, 48)]:
        rows = [(r0 + 8 * (m & 1) + i, c0 + 8 * (m >> 1)) for m in range(4) for i in range(8)]
        sw = [2 * orc.swizzle(r * 64 + c, B=3, M=3, S=3) for r, c in rows]
        assert _ways(orc, sw, 16) == (1, 4)
        plain = [2 * (r * 64 + c) for r, c in rows]
        assert _ways(orc, plain, 16) == (8, 32)


def test_bank_8byte_passes(orc):
    """"NVIDIA CuTe Swizzle": one operation serves at most 64 fp16 values of
    distinct columns, i.e. 128 bytes; more takes further passes, and that
    minimum is not a conflict.  A warp reading 32 consecutive 8-byte words
    (256 bytes) therefore takes two passes and has no conflict.  Reading
    down an 8-byte column of 128-byte rows puts each half-warp pass on one
    bank pair: 16 distinct words per bank in each of the two passes."""
    assert _ways(orc, [8 * l for l in range(32)], 8) == (1, 2)
    assert _ways(orc, [128 * l + 8 for l in range(32)], 8) == (16, 32)
    # the same 256 bytes as 4-byte accesses: one pass (two words per lane pair)
    assert _ways(orc, [4 * l for l in range(32)], 4) == (1, 1)


def test_bank_inactive_and_unaligned(orc):
    # inactive lanes do not count
    col = [4 * (r * 32) for r in range(32)]
    assert _ways(orc, col, 4, active=0x1)[0] == 1
    assert _ways(orc, col, 4, active=0)[0] == 0
    # a 4-byte access at byte 2 straddles words 0 and 1
    assert _ways(orc, [2, 130], 4) == (2, 2)


# -------------------------------------------------------- slice collision ---

def test_collision_truth_table(orc):
    """"cutlass 入门", section "swizzle 融入 layout 优化": for one (Z_i, Y_i)
    pair, C at Z_i is set exactly when both bits are active."""
    table = [tuple(int(v) for v in row) for row in read_golden("collision_truth_table.txt")]
    assert len(table) == 4
    B, M, S = 3, 2, 4
    for i in range(B):
        z, y = M + i, M + S + i
        for a_z, a_y, sw_z, c_z in table:
            A = (a_z << z) | (a_y << y)
            assert (orc.swizzle(A, B=B, M=M, S=S) >> z) & 1 == sw_z
            C = orc.slice_collision(A, B=B, M=M, S=S)
            assert (C >> z) & 1 == c_z
            assert C & ~(1 << z) == 0


@pytest.mark.parametrize("B,M,S", [(1, 0, 1), (2, 0, 2), (2, 1, 2), (2, 0, 3), (3, 0, 3),
                                   (2, 0, 1), (3, 0, 1), (3, 1, 2),
                                   (2, 0, -2), (3, 0, -1), (3, 1, -2)])
def test_collision_predicts_layout(orc, B, M, S):
    """Brute force: C == 0 exactly when the swizzle restricted to the slice is a
    plain layout (a sum of per-bit strides), on every mask A of the low bits."""
    nbits = B + M + abs(S) + 1
    for A in range(1 << nbits):
        C = orc.slice_collision(A, B=B, M=M, S=S)
        assert (C == 0) == orc.slice_is_layout(A, B=B, M=M, S=S), (A, C)


def test_dump_layout(orc):
    text = orc.dump_layout(32, 64, 4, B=5, M=0, S=6)
    lines = text.splitlines()
    assert len(lines) == 32
    entry = lines[10].split()[33]
    assert entry == f"683/{683 % 32}"
