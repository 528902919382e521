"""Negative SShift on the GPU, bit for bit against the oracle.

A negative shift reads the field at MBase and writes the field |S| bits above
it (the reading of "NVIDIA CuTe Swizzle"'s bit-diagram comment that the oracle
pins).  The read field can then sit below a 16-byte vector's lane bits while
the written one sits above them, so the relayout takes other paths than for a
positive shift: whole vectors (M >= log2 V), a fixed lane map when the map
stays inside a vector, cosets of whole vectors in registers (with a fixed lane
map when the written field starts inside the lanes), staged periods in shared
memory for ragged tiles, element by element.  The parameter grid below reaches each of them for every element
size."""
import numpy as np
import pytest

from gpu_util import empty_device, guards_intact, to_device, to_host, torch, void_dtype

pytestmark = pytest.mark.gpu

NEGATIVE = [(B, M, -s) for B in range(1, 6) for M in range(0, 5) for s in range(1, 8)]


@pytest.fixture(scope="module")
def swz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import xor_swizzle_movement_gb300 as m
    m.lib()
    return m


def _wtop(B, M, S):
    """Offsets close under the swizzle in aligned blocks of 2^wtop elements."""
    return M - S + B


def _run(swz, orc, host, n_tiles, rows, cols, esize, B, M, S, direction, src_off=0, dst_off=0, tma=False):
    _, src = to_device(host, src_off)
    full, dst = empty_device(host.nbytes, dst_off)
    fn = swz.swz_relayout_tma if tma else swz.swz_relayout
    fn(dst, src, n_tiles, rows, cols, esize, B, M, S, direction)
    torch.cuda.synchronize()
    want = orc.relayout(host, tile_elems=rows * cols, B=B, M=M, S=S, direction=direction)
    got = to_host(dst, host.dtype)
    assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), (esize, B, M, S, direction)
    assert guards_intact(full, dst_off, host.nbytes)


@pytest.mark.parametrize("esize", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("B,M,S", NEGATIVE)
def test_relayout_negative_shift(swz, orc, esize, B, M, S):
    """Three tiles of two closure blocks each, both directions."""
    from xor_swizzle_movement_gb300 import inputs
    period = 1 << _wtop(B, M, S)
    rows, cols, n_tiles = 2, period, 3
    host = inputs.random_bytes(n_tiles * rows * cols * esize, seed=40 + B * 100 + M * 10 - S).view(void_dtype(esize))
    for direction in (0, 1):
        _run(swz, orc, host, n_tiles, rows, cols, esize, B, M, S, direction)


@pytest.mark.parametrize("esize,mult,B,M,S,src_off,dst_off", [
    (1, 3, 1, 0, -1, 0, 0),     # 12-byte tiles: staged ragged tiles
    (1, 3, 2, 0, -1, 0, 0),     # 24-byte tiles
    (2, 5, 1, 0, -1, 0, 0),     # 40-byte tiles
    (1, 1, 1, 1, -1, 0, 0),     # 8-byte tiles: two per vector, fixed lane map
    (2, 2, 2, 0, -2, 2, 0),     # unaligned source: element by element
    (4, 3, 3, 1, -3, 0, 4),     # unaligned destination
    (8, 1, 2, 0, -5, 8, 8),
    (1, 2, 5, 0, -7, 1, 3),
])
def test_relayout_negative_shift_ragged_and_unaligned(swz, orc, esize, mult, B, M, S, src_off, dst_off):
    from xor_swizzle_movement_gb300 import inputs
    tile = mult << _wtop(B, M, S)
    n_tiles = 7
    host = inputs.random_bytes(n_tiles * tile * esize, seed=77 + mult).view(void_dtype(esize))
    for direction in (0, 1):
        _run(swz, orc, host, n_tiles, 1, tile, esize, B, M, S, direction, src_off, dst_off)


@pytest.mark.slow
@pytest.mark.parametrize("B,M,S", [(3, 3, -3),    # whole vectors move (M >= log2 8)
                                   (3, 0, -4),    # warp shuffles (cosets of 8 inside blocks of 32 vectors)
                                   (3, 1, -7),    # register cosets of 4 vectors
                                   (4, 2, -9),    # register cosets of 2 vectors, 8 per thread
                                   (4, 0, -9),    # register cosets of 8 vectors, one more read bit above the lanes
                                   (3, 0, -2),    # written field inside the lanes: warp shuffles after a lane map
                                   (16, 0, -2),   # register cosets with a lane map, 2^18-element blocks, 8 inverse steps
                                   (2, 0, -1)])   # the whole map inside one vector: fixed lane map
def test_relayout_negative_shift_64mib(swz, orc, B, M, S):
    """A 64 MiB uint16 buffer as one tile, every position, both directions,
    and forward then inverse gives the input back."""
    from xor_swizzle_movement_gb300 import inputs
    n = 1 << 25
    host = inputs.uint16_bits(n, seed=9)
    src = torch.from_numpy(host.view(np.int16).copy()).cuda()
    fwd, back = torch.empty_like(src), torch.empty_like(src)
    swz.swz_relayout(fwd, src, 1, 1, n, 2, B, M, S, 0)
    swz.swz_relayout(back, fwd, 1, 1, n, 2, B, M, S, 1)
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    want = orc.relayout(host, tile_elems=n, B=B, M=M, S=S, direction=0)
    assert np.array_equal(fwd.cpu().numpy().view(np.uint16), want)


# Negative shifts that split vectors, at a few MiB (many CTAs, and an odd
# number of closure blocks so that the last CTA or warp is partly idle): sets
# that reach every path, with the path each direction takes (several with
# overlapping fields, |S| < B).
COSETS = [
    # esize, B, M, S
    (1, 1, 0, -4),          # warp shuffles
    (1, 2, 0, -5),          # warp shuffles
    (1, 3, 0, -6),          # warp shuffles
    (1, 5, 0, -4),          # warp shuffles
    (1, 4, 0, -9),          # register cosets U 1 g 4
    (1, 3, 1, -3),          # warp shuffles
    (2, 2, 0, -3),          # warp shuffles
    (2, 1, 0, -5),          # warp shuffles
    (2, 4, 1, -2),          # warp shuffles
    (4, 1, 0, -2),          # warp shuffles
    (4, 3, 0, -2),          # warp shuffles
    (8, 2, 0, -1),          # warp shuffles
    (1, 1, 3, -1),          # warp shuffles
    (2, 6, 0, -5),          # register cosets U 2 g 3
    (2, 3, 2, -3),          # warp shuffles
    (1, 4, 3, -4),          # register cosets U 8 g 1 SB 3
    (2, 4, 1, -4),          # warp shuffles, 64-vector blocks
    (1, 4, 2, -5),          # register cosets U 4 g 2 SB 2
    (2, 5, 0, -5),          # register cosets U 2 g 3 SB 1
    (1, 5, 1, -6),          # register cosets U 2 g 3 SB 1
    (1, 2, 0, -4),          # warp shuffles
    (1, 3, 0, -4),          # warp shuffles
    (1, 4, 0, -4),          # warp shuffles
    (2, 1, 0, -3),          # warp shuffles
    (4, 2, 0, -2),          # warp shuffles
    (2, 4, 0, -3),          # warp shuffles
    (1, 5, 1, -3),          # warp shuffles
    (1, 3, 2, -2),          # warp shuffles
    (2, 3, 0, -4),          # warp shuffles
    (4, 2, 0, -3),          # warp shuffles
    (8, 1, 0, -2),          # warp shuffles
    (4, 1, 0, -4),          # warp shuffles
    (1, 1, 0, -5),          # warp shuffles
    (2, 2, 0, -4),          # warp shuffles
    (1, 2, 0, -3),          # warp shuffles after a lane map
    (1, 3, 0, -3),          # warp shuffles after a lane map
    (1, 4, 0, -3),          # warp shuffles after a lane map
    (1, 9, 0, -3),          # lane-map cosets g 3 block stores; inverse: lane-map cosets g 3
    (2, 2, 1, -1),          # warp shuffles after a lane map
    (2, 3, 0, -2),          # warp shuffles after a lane map
    (2, 12, 0, -1),         # lane-map cosets g 1 block stores; inverse: lane-map cosets g 1
    (4, 2, 0, -1),          # warp shuffles after a lane map
    (4, 7, 0, -1),          # warp shuffles, 64-vector blocks after a lane map
    (2, 4, 0, -2),          # warp shuffles after a lane map
    (1, 5, 0, -3),          # warp shuffles after a lane map
    (1, 5, 0, -5),          # register cosets U 1 g 4
    (2, 5, 0, -4),          # warp shuffles, 64-vector blocks
    (1, 5, 1, -4),          # warp shuffles, 64-vector blocks
    (1, 1, 0, -9),          # register cosets U 1 g 1
    (1, 7, 0, -3),          # lane-map cosets g 3 block stores; inverse: lane-map cosets g 3
    (2, 1, 0, -8),          # warp shuffles, 64-vector blocks
    (2, 7, 0, -2),          # warp shuffles, 64-vector blocks after a lane map
    (4, 1, 0, -7),          # warp shuffles, 64-vector blocks
    (8, 1, 0, -6),          # warp shuffles, 64-vector blocks
]

# Sets that stay on the register coset kernels (their sources leave the
# destination's block of 64 vectors): one per instantiation.
COSETS_REG = [
    # esize, B, M, S
    (1, 1, 0, -10),         # register cosets U 1 g 1
    (1, 2, 0, -9),          # register cosets U 1 g 2
    (1, 3, 0, -8),          # register cosets U 1 g 3
    (1, 4, 0, -7),          # register cosets U 1 g 4
    (1, 7, 0, -4),          # register cosets U 1 g 4 block stores; inverse: register cosets U 1 g 4
    (2, 1, 0, -9),          # register cosets U 2 g 1
    (2, 2, 0, -8),          # register cosets U 2 g 2
    (2, 3, 0, -7),          # register cosets U 2 g 3
    (2, 7, 0, -3),          # register cosets U 2 g 3 block stores; inverse: register cosets U 2 g 3
    (2, 5, 0, -5),          # register cosets U 2 g 3 SB 1
    (4, 1, 0, -8),          # register cosets U 4 g 1
    (4, 2, 0, -7),          # register cosets U 4 g 2
    (4, 7, 0, -2),          # register cosets U 4 g 2 block stores; inverse: register cosets U 4 g 2
    (4, 4, 0, -5),          # register cosets U 4 g 2 SB 2
    (8, 1, 0, -7),          # register cosets U 8 g 1
    (8, 7, 0, -1),          # register cosets U 8 g 1 block stores; inverse: register cosets U 8 g 1
    (8, 3, 0, -5),          # register cosets U 8 g 1 SB 2
    (8, 4, 0, -4),          # register cosets U 8 g 1 SB 3
    (4, 8, 0, -1),          # lane-map cosets g 1 block stores; inverse: lane-map cosets g 1
    (2, 8, 0, -2),          # lane-map cosets g 2 block stores; inverse: lane-map cosets g 2
    (1, 8, 0, -3),          # lane-map cosets g 3 block stores; inverse: lane-map cosets g 3
]


@pytest.mark.parametrize("esize,B,M,S", COSETS + COSETS_REG)
def test_relayout_cosets_ragged_grid(swz, orc, esize, B, M, S):
    from xor_swizzle_movement_gb300 import inputs
    block = 1 << _wtop(B, M, S)
    n_blocks = max(1, (6 << 20) // (block * esize)) | 1
    tile = block * (n_blocks if n_blocks < 8 else 1)
    n_tiles = (block * n_blocks) // tile
    host = inputs.random_bytes(n_tiles * tile * esize, seed=500 + esize * 37 + B * 5 - S).view(void_dtype(esize))
    for direction in (0, 1):
        _run(swz, orc, host, n_tiles, 1, tile, esize, B, M, S, direction)


@pytest.mark.parametrize("esize,B,M,S", [(1, 7, 0, -4), (2, 7, 0, -3), (4, 7, 0, -2), (8, 7, 0, -1), (4, 8, 0, -1)])
@pytest.mark.parametrize("src_off,dst_off", [(16, 48), (0, 16), (16, 0)])
def test_relayout_cosets_block_16_byte_aligned(swz, orc, esize, B, M, S, src_off, dst_off):
    """Cosets whose destination side is an aligned block (stored with 32-byte
    accesses on a 32-byte aligned destination), on pointers 16- but not 32-byte
    aligned: the kernels keep 16-byte stores."""
    from xor_swizzle_movement_gb300 import inputs
    block = 1 << _wtop(B, M, S)
    n_tiles = 1001
    host = inputs.random_bytes(n_tiles * block * esize, seed=900 + esize).view(void_dtype(esize))
    for direction in (0, 1):
        _run(swz, orc, host, n_tiles, 1, block, esize, B, M, S, direction, src_off, dst_off)


@pytest.mark.parametrize("esize,rows,cols,te,B,M,S", [
    (2, 64, 4096, 8192, 3, 3, -4),    # M >= log2 8: 16-byte vectors land whole
    (2, 64, 4096, 8192, 2, 1, -3),    # M < log2 8: element by element
    (4, 96, 520, 1040, 1, 0, -2),     # ragged matrix, fp32
    (1, 256, 384, 4096, 3, 0, -5),    # bytes
    (8, 48, 80, 64, 2, 1, -1),        # fp64, overlapping fields
])
def test_transpose_relayout_negative_shift(swz, orc, esize, rows, cols, te, B, M, S):
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.random_bytes(rows * cols * esize, seed=3 + esize).view(void_dtype(esize)).reshape(rows, cols)
    _, src = to_device(host)
    full, dst = empty_device(host.nbytes)
    swz.swz_transpose_relayout(dst, src, rows, cols, esize, te, B, M, S)
    torch.cuda.synchronize()
    want = orc.transpose_relayout(host, tile_elems=te, B=B, M=M, S=S)
    assert np.array_equal(to_host(dst, host.dtype).view(np.uint8), want.view(np.uint8))
    assert guards_intact(full, 0, host.nbytes)


def test_relayout_tma_negative_shift_runs_register_kernels(swz, orc):
    """No tensor-map swizzle mode has a negative shift: the TMA entry point
    reports path 0 and runs the register kernels, with the oracle's result."""
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.random_bytes(64 * 64 * 2 * 16, seed=5).view(np.uint16)
    _, src = to_device(host)
    _, dst = empty_device(host.nbytes)
    assert swz.swz_relayout_tma_path(dst, src, 16, 64, 64, 2, 3, 3, -3, 0) == 0
    _run(swz, orc, host, 16, 64, 64, 2, 3, 3, -3, 0, tma=True)


def test_slice_collision_batch_negative_shift(swz, orc):
    rng = np.random.default_rng(11)
    A = rng.integers(0, 1 << 40, 4096, dtype=np.int64)
    dA = torch.from_numpy(A).cuda()
    for B, M, S in [(3, 2, -4), (2, 0, -1), (5, 1, -9)]:
        C = torch.empty_like(dA)
        swz.swz_slice_collision_batch(dA, A.size, B, M, S, C)
        torch.cuda.synchronize()
        got = C.cpu().numpy().view(np.uint64)
        want = np.array([orc.slice_collision(int(a), B=B, M=M, S=S) for a in A], dtype=np.uint64)
        assert np.array_equal(got, want)


NEG_SWEEP = [(esize, B, M, -s) for esize, lv in ((2, 3), (1, 4)) for B in range(1, 6) for M in range(lv)
             for s in range(1, 6)]


@pytest.fixture(scope="module")
def gib_bytes():
    """1 GiB of random bytes (seed 4), on the GPU: the bench's negative-shift sweep buffer."""
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    return torch.randint(0, 256, (1 << 30,), dtype=torch.uint8, device="cuda", generator=g)


@pytest.mark.slow
@pytest.mark.parametrize("esize,B,M,S", NEG_SWEEP)
def test_negative_sweep_1gib_every_position(swz, orc, gib_bytes, esize, B, M, S):
    """Every negative set the bench's sweep times (uint16 and int8, B 1..5, M
    below log2 V, S -1..-5), on its 1 GiB buffer as one tile and in its launch
    configuration, compared at every position in both directions.  The map
    reads and writes only offset bits below M + |S| + B <= 13, so the oracle's
    map of the first 2^16 offsets, repeated on every 2^16-element block, is the
    whole map; torch index operations apply it.  The oracle's map at 2^14
    random global offsets checks the repetition, and forward then inverse must
    give the input back."""
    period = 1 << 16
    n = (1 << 30) // esize
    dt = torch.int16 if esize == 2 else torch.uint8
    src = gib_bytes
    fwd, back = torch.empty_like(src), torch.empty_like(src)
    swz.swz_relayout(fwd, src, 1, 1, n, esize, B, M, S, 0)
    swz.swz_relayout(back, fwd, 1, 1, n, esize, B, M, S, 1)
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    perm = orc.relayout_positions(np.arange(period, dtype=np.int64), tile_elems=n, B=B, M=M, S=S)
    assert np.array_equal(np.sort(perm), np.arange(period))
    tp = torch.from_numpy(perm).cuda()
    s2 = src.view(dt).view(-1, period)
    want_fwd = torch.empty_like(s2).index_copy_(1, tp, s2)       # dst[sw(i)] = src[i]
    assert torch.equal(fwd.view(dt).view(-1, period), want_fwd)
    del want_fwd
    inv = torch.empty_like(src)
    swz.swz_relayout(inv, src, 1, 1, n, esize, B, M, S, 1)
    want_inv = s2.index_select(1, tp)                              # dst[i] = src[sw(i)]
    assert torch.equal(inv.view(dt).view(-1, period), want_inv)
    del want_inv, inv
    rng = np.random.default_rng(esize * 1000 + B * 100 + M * 10 - S)
    idx = np.sort(rng.choice(n, 1 << 14, replace=False)).astype(np.int64)
    pos = orc.relayout_positions(idx, tile_elems=n, B=B, M=M, S=S)
    ti = torch.from_numpy(idx).cuda()
    assert torch.equal(fwd.view(dt)[torch.from_numpy(pos).cuda()], src.view(dt)[ti])
