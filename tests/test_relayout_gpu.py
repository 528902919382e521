"""GPU relayout (swz_relayout through the C ABI) against the CPU oracle.

Bit-exact comparisons: relayout is a permutation of raw element bits.
Inputs are the seeded generators of xor_swizzle_movement_gb300.inputs."""
import itertools

import numpy as np
import pytest

from gpu_util import empty_device, guards_intact, to_device, to_host, torch, void_dtype

pytestmark = pytest.mark.gpu

SWEEP = [(B, M, S) for B in range(1, 6) for M in range(0, 5) for S in range(B, 8)]


@pytest.fixture(scope="module")
def swz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import xor_swizzle_movement_gb300 as m
    m.lib()
    return m


def run_relayout(swz, host, n_tiles, rows, cols, esize, B, M, S, direction, src_off=0, dst_off=0):
    nbytes = host.nbytes
    _, src = to_device(host, src_off)
    full, dst = empty_device(nbytes, dst_off)
    swz.swz_relayout(dst, src, n_tiles, rows, cols, esize, B, M, S, direction)
    torch.cuda.synchronize()
    assert guards_intact(full, dst_off, nbytes)
    return to_host(dst, host.dtype)


def test_small_fp16_tiles_sw333(swz, orc):
    """256 tiles of 64 x 64 16-bit elements, Swizzle<3,3,3>, forward then inverse."""
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.uint16_bits(256 * 64 * 64, seed=0)
    fwd = run_relayout(swz, host, 256, 64, 64, 2, 3, 3, 3, 0)
    assert np.array_equal(fwd, orc.relayout(host, tile_elems=4096, B=3, M=3, S=3, direction=0))
    inv = run_relayout(swz, host, 256, 64, 64, 2, 3, 3, 3, 1)
    assert np.array_equal(inv, orc.relayout(host, tile_elems=4096, B=3, M=3, S=3, direction=1))
    back = run_relayout(swz, fwd, 256, 64, 64, 2, 3, 3, 3, 1)
    assert np.array_equal(back, host)


@pytest.mark.slow
def test_bf16_tiles_sw343_full(swz, orc):
    """4096 bf16 tiles of 128 x 64 (64 MiB), Swizzle<3,4,3>, both directions."""
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.bf16_normal(4096 * 128 * 64, seed=1)
    for direction in (0, 1):
        got = run_relayout(swz, host, 4096, 128, 64, 2, 3, 4, 3, direction)
        want = orc.relayout(host, tile_elems=128 * 64, B=3, M=4, S=3, direction=direction)
        assert np.array_equal(got, want)


@pytest.mark.parametrize("B,M,S", SWEEP)
def test_uint16_sweep(swz, orc, B, M, S):
    """Every (B, M, S) of the sweep on one 2^20-element uint16 buffer."""
    from xor_swizzle_movement_gb300 import inputs
    n = 1 << 20
    host = inputs.random_bytes(2 * n, seed=4).view(np.uint16)
    for direction in (0, 1):
        got = run_relayout(swz, host, 1, 1, n, 2, B, M, S, direction)
        want = orc.relayout(host, tile_elems=n, B=B, M=M, S=S, direction=direction)
        assert np.array_equal(got, want), direction


@pytest.fixture(scope="module")
def gib_u16():
    """The 1 GiB uint16 buffer of the sweep (random bytes, seed 4), on the GPU."""
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    return torch.randint(0, 256, (1 << 30,), dtype=torch.uint8, device="cuda", generator=g)


@pytest.mark.slow
@pytest.mark.parametrize("B,M,S", SWEEP)
def test_uint16_sweep_1gib_every_position(swz, orc, gib_u16, B, M, S):
    """The 1 GiB uint16 buffer as one tile, every (B, M, S) of the sweep, in
    the launch configuration the bench times, compared at every one of the
    2^29 positions in both directions.  The swizzle reads and writes only
    offset bits below B + M + S <= 16, so the oracle's map of the first 2^16
    offsets, repeated on every 2^16-element block, is the whole map; torch
    index operations apply it to build the expected buffers.  The oracle's
    map at 2^16 random global offsets checks that repetition, and forward
    then inverse must give the input back."""
    n, period = 1 << 29, 1 << 16
    src = gib_u16
    fwd = torch.empty_like(src)
    back = torch.empty_like(src)
    swz.swz_relayout(fwd, src, 1, 1, n, 2, B, M, S, 0)
    swz.swz_relayout(back, fwd, 1, 1, n, 2, B, M, S, 1)
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    perm = orc.relayout_positions(np.arange(period, dtype=np.int64), tile_elems=n, B=B, M=M, S=S)
    assert np.array_equal(np.sort(perm), np.arange(period))
    tp = torch.from_numpy(perm).cuda()
    s2 = src.view(torch.int16).view(-1, period)
    want_fwd = torch.empty_like(s2).index_copy_(1, tp, s2)       # dst[sw(i)] = src[i]
    assert torch.equal(fwd.view(torch.int16).view(-1, period), want_fwd)
    del want_fwd
    inv = torch.empty_like(src)
    swz.swz_relayout(inv, src, 1, 1, n, 2, B, M, S, 1)
    want_inv = s2.index_select(1, tp)                              # dst[i] = src[sw(i)]
    assert torch.equal(inv.view(torch.int16).view(-1, period), want_inv)
    del want_inv, inv
    rng = np.random.default_rng(B * 100 + M * 10 + S)
    idx = np.sort(rng.choice(n, 1 << 16, replace=False)).astype(np.int64)
    pos = orc.relayout_positions(idx, tile_elems=n, B=B, M=M, S=S)
    ti = torch.from_numpy(idx).cuda()
    assert torch.equal(fwd.view(torch.int16)[torch.from_numpy(pos).cuda()], src.view(torch.int16)[ti])


@pytest.mark.slow
def test_int8_tiles_sw525_full(swz, orc):
    """int8 tiles of 64 x 128 (1 GiB), Swizzle<5,2,5> (4-byte groups)."""
    from xor_swizzle_movement_gb300 import inputs
    n_tiles = (1 << 30) // (64 * 128)
    host = inputs.random_bytes(1 << 30, seed=4)
    for direction in (0, 1):
        got = run_relayout(swz, host, n_tiles, 64, 128, 1, 5, 2, 5, direction)
        want = orc.relayout(host, tile_elems=64 * 128, B=5, M=2, S=5, direction=direction)
        assert np.array_equal(got, want), direction


GRID_BMS = [(3, 0, 1), (3, 1, 2), (2, 0, 1), (4, 1, 1), (5, 0, 2), (3, 3, 3), (2, 5, 3), (1, 0, 1),
            (4, 0, 4), (0, 2, 3), (5, 2, 5), (2, 2, 6)]


@pytest.mark.parametrize("esize", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("B,M,S", GRID_BMS)
def test_esize_grid(swz, orc, esize, B, M, S):
    """All element sizes, including S < B (not self-inverse), several tiles."""
    from xor_swizzle_movement_gb300 import inputs
    tile = 1 << (B + M + S)
    rows, cols = (tile // 8, 8) if tile >= 8 else (1, tile)
    n_tiles = 3
    host = inputs.random_bytes(n_tiles * tile * esize, seed=4).view(void_dtype(esize))
    for direction in (0, 1):
        got = run_relayout(swz, host, n_tiles, rows, cols, esize, B, M, S, direction)
        want = orc.relayout(host, tile_elems=tile, B=B, M=M, S=S, direction=direction)
        assert got.tobytes() == want.tobytes(), direction


@pytest.mark.parametrize("esize,rows,cols,B,M,S,n_tiles", [
    (2, 3, 4, 2, 0, 1, 5),      # 24-byte tiles: element-by-element path
    (4, 5, 16, 2, 1, 2, 7),     # 320-byte tiles, period 32 does not divide 80
    (2, 24, 64, 3, 3, 3, 9),    # period 512 does not divide 1536: tile-local offsets
    (1, 3, 64, 3, 2, 3, 11),    # tile-local offsets, 192-byte tiles
    (8, 6, 8, 2, 1, 3, 5),      # 384-byte tiles, period 64 does not divide 48
    (16, 3, 4, 2, 0, 2, 3),     # 16-byte elements, tile-local
])
def test_ragged_tiles(swz, orc, esize, rows, cols, B, M, S, n_tiles):
    from xor_swizzle_movement_gb300 import inputs
    tile = rows * cols
    host = inputs.random_bytes(n_tiles * tile * esize, seed=7).view(void_dtype(esize))
    for direction in (0, 1):
        got = run_relayout(swz, host, n_tiles, rows, cols, esize, B, M, S, direction)
        want = orc.relayout(host, tile_elems=tile, B=B, M=M, S=S, direction=direction)
        assert got.tobytes() == want.tobytes()


@pytest.mark.parametrize("esize,tile,B,M,S", [
    (1, 2, 1, 0, 1), (1, 4, 1, 0, 1), (1, 4, 2, 0, 1), (1, 8, 1, 0, 2), (1, 8, 2, 1, 1), (1, 8, 3, 0, 1),
    (2, 2, 1, 0, 3), (2, 4, 2, 0, 1), (2, 4, 1, 1, 1), (4, 2, 1, 0, 1), (8, 1, 0, 0, 1)])
@pytest.mark.parametrize("n_tiles", [4096, 4099])
def test_tiles_smaller_than_a_vector(swz, orc, esize, tile, B, M, S, n_tiles):
    """Tiles of 1 to 8 bytes: whole tiles inside every 16-byte vector (a fixed
    lane permutation), and a count that leaves a partial vector (element path)."""
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.random_bytes(n_tiles * tile * esize, seed=9).view(void_dtype(esize))
    for direction in (0, 1):
        got = run_relayout(swz, host, n_tiles, 1, tile, esize, B, M, S, direction)
        want = orc.relayout(host, tile_elems=tile, B=B, M=M, S=S, direction=direction)
        assert got.tobytes() == want.tobytes(), direction


@pytest.mark.parametrize("esize,tile,B,M,S", [
    (1, 24, 2, 0, 1), (1, 40, 3, 0, 2), (1, 12, 2, 0, 3), (1, 1000, 3, 0, 3), (2, 12, 2, 0, 1),
    (2, 20, 2, 0, 2), (2, 76, 2, 0, 3), (4, 6, 1, 0, 1), (4, 10, 1, 0, 1), (4, 30, 1, 0, 5),
    (8, 3, 0, 0, 1), (8, 10, 1, 0, 2), (8, 6, 1, 0, 1),
    # groups of 2^M elements gathered as units of 2, 4 or 8 bytes
    (1, 40, 2, 1, 2), (1, 24, 1, 2, 3), (2, 12, 1, 1, 2), (1, 56, 0, 3, 1), (4, 14, 0, 1, 1),
    (2, 28, 1, 1, 3),
    # S < B: the forward gathers through the exact inverse
    (1, 24, 2, 1, 1), (2, 20, 2, 0, 1)])
@pytest.mark.parametrize("n_tiles", [1, 1000, 4099])
def test_ragged_tiles_staged(swz, orc, esize, tile, B, M, S, n_tiles):
    """Tiles whose byte size is not a multiple of 16 (aligned pointers): whole
    tiles staged in shared memory in blocks of lcm(tile bytes, 16) x k bytes,
    including a last block that is partial and not a multiple of 16 bytes."""
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.random_bytes(n_tiles * tile * esize, seed=10).view(void_dtype(esize))
    for direction in (0, 1):
        got = run_relayout(swz, host, n_tiles, 1, tile, esize, B, M, S, direction)
        want = orc.relayout(host, tile_elems=tile, B=B, M=M, S=S, direction=direction)
        assert got.tobytes() == want.tobytes(), direction


@pytest.mark.parametrize("esize,tile,B,M,S", [
    (1, 24, 2, 0, 1),     # 8-byte periods in 24-byte tiles
    (1, 40, 1, 1, 1),     # 8-element periods, groups of 2 bytes
    (2, 12, 1, 0, 1),     # 4-element periods in 24-byte tiles
    (1, 24, 1, 0, -2),    # negative shift: 8-byte closure blocks, cosets with a lane map
    (2, 12, 1, 0, -1),    # negative shift inside one vector
    (8, 3, 0, 0, 1)])     # B = 0: a copy
@pytest.mark.parametrize("n_tiles", [1 << 18, (1 << 18) + 2])
def test_ragged_tiles_of_whole_periods(swz, orc, esize, tile, B, M, S, n_tiles):
    """Tiles that are not whole 16-byte vectors but hold whole swizzle periods:
    the swizzle is the same on whole-buffer offsets, and a buffer of whole
    vectors runs as one tile (several MiB, many CTAs)."""
    from xor_swizzle_movement_gb300 import inputs
    if (n_tiles * tile * esize) % 16:
        n_tiles += 1
    host = inputs.random_bytes(n_tiles * tile * esize, seed=12).view(void_dtype(esize))
    for direction in (0, 1):
        got = run_relayout(swz, host, n_tiles, 1, tile, esize, B, M, S, direction)
        want = orc.relayout(host, tile_elems=tile, B=B, M=M, S=S, direction=direction)
        assert got.tobytes() == want.tobytes(), direction


@pytest.mark.parametrize("esize", [1, 2, 4, 8])
def test_misaligned_pointers(swz, orc, esize):
    """Pointers aligned to the element size but not to 16 bytes."""
    from xor_swizzle_movement_gb300 import inputs
    B, M, S, rows, cols, n_tiles = 3, 1, 3, 16, 8, 6
    host = inputs.random_bytes(n_tiles * rows * cols * esize, seed=8).view(void_dtype(esize))
    got = run_relayout(swz, host, n_tiles, rows, cols, esize, B, M, S, 0, src_off=esize, dst_off=3 * esize)
    want = orc.relayout(host, tile_elems=rows * cols, B=B, M=M, S=S, direction=0)
    assert got.tobytes() == want.tobytes()


def test_empty_and_errors(swz):
    _, a = empty_device(4096)
    _, b = empty_device(4096)
    # empty requests launch nothing and succeed
    swz.swz_relayout(b, a, 0, 64, 64, 2, 3, 3, 3, 0)
    swz.swz_relayout(b, a, 5, 0, 64, 2, 3, 3, 3, 0)
    cases = [
        (dict(n_tiles=1, rows=3, cols=4, esize=2, B=2, M=2, S=2), swz.SWZ_ERR_SHAPE),  # 12 % 16 != 0
        (dict(n_tiles=1, rows=8, cols=8, esize=2, B=3, M=0, S=0), swz.SWZ_ERR_PARAM),  # S = 0
        (dict(n_tiles=1, rows=8, cols=8, esize=3, B=3, M=0, S=3), swz.SWZ_ERR_PARAM),  # esize
        (dict(n_tiles=1, rows=8, cols=8, esize=2, B=3, M=0, S=-6), swz.SWZ_ERR_SHAPE),  # 64 % 2^9 != 0
        (dict(n_tiles=1, rows=8, cols=8, esize=2, B=3, M=0, S=-33), swz.SWZ_ERR_PARAM),
        (dict(n_tiles=-1, rows=8, cols=8, esize=2, B=3, M=0, S=3), swz.SWZ_ERR_SHAPE),
    ]
    for kw, status in cases:
        with pytest.raises(swz.SwzError) as e:
            swz.swz_relayout(b, a, kw["n_tiles"], kw["rows"], kw["cols"], kw["esize"], kw["B"], kw["M"],
                             kw["S"], 0)
        assert e.value.status == status, kw
    with pytest.raises(swz.SwzError) as e:
        swz.swz_relayout(a, a, 1, 8, 8, 2, 3, 0, 3, 0)
    assert e.value.status == swz.SWZ_ERR_ALIAS
    with pytest.raises(swz.SwzError) as e:
        swz.swz_relayout(a[1:], b, 1, 8, 8, 2, 3, 0, 3, 0)
    assert e.value.status == swz.SWZ_ERR_ALIGN


def test_host_buffers_through_the_device_address_space(swz, orc):
    """Pinned host memory is addressable by the kernels: a forward relayout
    reads a pinned host buffer and the inverse writes one, and the result
    matches the oracle."""
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.uint16_bits(64 * 64 * 64, seed=6)
    h_src = torch.from_numpy(host.view(np.int16).copy()).pin_memory()
    h_back = torch.zeros_like(h_src).pin_memory()
    phys = torch.empty(h_src.numel(), dtype=torch.int16, device="cuda")
    swz.swz_relayout(phys, h_src.data_ptr(), 64, 64, 64, 2, 3, 3, 3, 0)
    swz.swz_relayout(h_back.data_ptr(), phys, 64, 64, 64, 2, 3, 3, 3, 1)
    torch.cuda.synchronize()
    want = orc.relayout(host, tile_elems=4096, B=3, M=3, S=3, direction=0)
    assert np.array_equal(phys.cpu().numpy().view(np.uint16), want)
    assert np.array_equal(h_back.numpy().view(np.uint16), host)


@pytest.mark.parametrize("esize,rows,cols,bms", [
    (1, 64, 128, (5, 2, 5)),    # the int8 tiles, lanes XOR-ed
    (2, 64, 64, (3, 3, 3)),     # 16-bit, lanes fixed
    (2, 3, 8, (2, 1, 3)),       # 48-byte tiles, period 64 elements: tile-local offsets
    (4, 5, 8, (2, 1, 1)),       # S < B, 160-byte tiles: tile-local offsets, general lane map
])
def test_host_buffers_larger_than_the_link_grid(swz, orc, esize, rows, cols, bms):
    """On host buffers the library caps the grid at 4 CTAs per SM and strides
    over the buffer; 64 MiB takes several strides.  Forward reads a pinned
    host buffer, inverse writes one; both match the oracle."""
    from xor_swizzle_movement_gb300 import inputs
    tile_bytes = rows * cols * esize
    n_tiles = (64 << 20) // tile_bytes
    host = inputs.random_bytes(n_tiles * tile_bytes, seed=8)
    h_src = torch.from_numpy(host.copy()).pin_memory()
    h_back = torch.zeros_like(h_src).pin_memory()
    phys = torch.empty(h_src.numel(), dtype=torch.uint8, device="cuda")
    B, M, S = bms
    swz.swz_relayout(phys, h_src.data_ptr(), n_tiles, rows, cols, esize, B, M, S, 0)
    swz.swz_relayout(h_back.data_ptr(), phys, n_tiles, rows, cols, esize, B, M, S, 1)
    torch.cuda.synchronize()
    view = {1: np.uint8, 2: np.uint16, 4: np.uint32}[esize]
    want = orc.relayout(host.view(view), tile_elems=rows * cols, B=B, M=M, S=S, direction=0)
    assert np.array_equal(phys.cpu().numpy().view(view), want)
    assert np.array_equal(h_back.numpy(), host)


@pytest.mark.parametrize("esize,src_off,dst_off", [
    (1, 1, 0), (1, 0, 7), (1, 3, 13), (2, 2, 0), (2, 0, 6), (2, 10, 14), (4, 4, 0), (4, 8, 12), (8, 8, 0), (8, 0, 8),
])
@pytest.mark.parametrize("rows,cols,bms,n_tiles", [
    (64, 64, (3, 3, 3), 9),     # the 16-bit config tile: tiles of whole vectors
    (64, 128, (5, 2, 5), 5),    # the int8 config tile
    (24, 64, (3, 3, 3), 3),     # period 512 does not divide 1536: tile-local offsets
    (8, 8, (2, 0, 1), 5),       # general lane map for 1- and 2-byte elements
    (1, 16, (1, 0, 1), 1),      # one or a few vectors: the buffer's first and last vectors coincide
    (1, 1 << 16, (5, 0, 11), 1),  # one large tile
    (3, 4, (2, 0, 1), 1001),    # ragged tiles: the staged kernel
    (1, 2, (1, 0, 1), 513),     # tiny tiles: the staged kernel
    (8, 16, (3, 0, -4), 33),    # a negative shift that splits vectors: staged blocks of 128 elements
    (2, 8, (0, 0, 1), 100),     # B = 0: a plain copy
    (6, 464, (0, 3, 2), 34),    # B = 0 with M = 3
])
def test_relayout_unaligned_pointers(swz, orc, esize, src_off, dst_off, rows, cols, bms, n_tiles):
    """Pointers aligned to the element size but not to 16 bytes.  Tiles of
    whole 16-byte vectors run the vector kernel on two aligned source chunks
    per vector and aligned destination chunks assembled across lanes; other
    tiles run the staged kernel at the pointers' offsets within their 16-byte
    chunks.  Both directions against the oracle; the guard bytes around the
    destination stay untouched."""
    from xor_swizzle_movement_gb300 import inputs
    B, M, S = bms
    host = inputs.random_bytes(n_tiles * rows * cols * esize, seed=21 + esize).view(void_dtype(esize))
    _, src = to_device(host, src_off)
    for direction in (0, 1):
        full, dst = empty_device(host.nbytes, dst_off)
        swz.swz_relayout(dst, src, n_tiles, rows, cols, esize, B, M, S, direction)
        torch.cuda.synchronize()
        want = orc.relayout(host, tile_elems=rows * cols, B=B, M=M, S=S, direction=direction)
        assert np.array_equal(to_host(dst, host.dtype).view(np.uint8), want.view(np.uint8)), direction
        assert guards_intact(full, dst_off, host.nbytes)


@pytest.mark.slow
@pytest.mark.parametrize("src_off,dst_off", [(2, 0), (0, 6), (10, 4)])
def test_relayout_unaligned_64mib(swz, orc, src_off, dst_off):
    """64 MiB of 16-bit 64 x 64 tiles under Swizzle<3,3,3> with pointers off
    16-byte alignment (four vectors per thread, many warps), both directions."""
    from xor_swizzle_movement_gb300 import inputs
    n_tiles = (64 << 20) // 8192
    host = inputs.uint16_bits(n_tiles * 4096, seed=31)
    _, src = to_device(host, src_off)
    for direction in (0, 1):
        full, dst = empty_device(host.nbytes, dst_off)
        swz.swz_relayout(dst, src, n_tiles, 64, 64, 2, 3, 3, 3, direction)
        torch.cuda.synchronize()
        want = orc.relayout(host, tile_elems=4096, B=3, M=3, S=3, direction=direction)
        assert np.array_equal(to_host(dst, np.uint16), want), direction
        assert guards_intact(full, dst_off, host.nbytes)


@pytest.mark.parametrize("src_off,dst_off", [(2, 6), (0, 10), (14, 0)])
def test_relayout_unaligned_tile_local_two_per_thread(swz, orc, src_off, dst_off):
    """About 700 000 vectors (two per thread on this GPU's grid), tiles of
    24 x 64 16-bit elements under Swizzle<3,4,3> (period 1024 elements does not
    divide the 1536-element tile: tile-local offsets), a last warp that is only
    partly used, pointers off 16-byte alignment; both directions."""
    from xor_swizzle_movement_gb300 import inputs
    n_tiles, rows, cols = 3647, 24, 64
    host = inputs.uint16_bits(n_tiles * rows * cols, seed=33)
    _, src = to_device(host, src_off)
    for direction in (0, 1):
        full, dst = empty_device(host.nbytes, dst_off)
        swz.swz_relayout(dst, src, n_tiles, rows, cols, 2, 3, 4, 3, direction)
        torch.cuda.synchronize()
        want = orc.relayout(host, tile_elems=rows * cols, B=3, M=4, S=3, direction=direction)
        assert np.array_equal(to_host(dst, np.uint16), want), direction
        assert guards_intact(full, dst_off, host.nbytes)


@pytest.mark.parametrize("src_off,dst_off", [(2, 0), (0, 6)])
def test_host_buffers_off_16_byte_alignment(swz, orc, src_off, dst_off):
    """Pinned host buffers whose pointers are off 16-byte alignment: the
    forward relayout reads the host buffer, the inverse writes one."""
    from xor_swizzle_movement_gb300 import inputs
    n_tiles = 512
    host = inputs.uint16_bits(n_tiles * 4096, seed=34)
    h_src = torch.zeros(host.nbytes + 16, dtype=torch.uint8).pin_memory()
    h_src[src_off:src_off + host.nbytes].copy_(torch.from_numpy(host.view(np.uint8)))
    h_back = torch.zeros(host.nbytes + 16, dtype=torch.uint8).pin_memory()
    phys = torch.empty(host.nbytes, dtype=torch.uint8, device="cuda")
    swz.swz_relayout(phys, h_src.data_ptr() + src_off, n_tiles, 64, 64, 2, 3, 3, 3, 0)
    swz.swz_relayout(h_back.data_ptr() + dst_off, phys, n_tiles, 64, 64, 2, 3, 3, 3, 1)
    torch.cuda.synchronize()
    want = orc.relayout(host, tile_elems=4096, B=3, M=3, S=3, direction=0)
    assert np.array_equal(phys.cpu().numpy().view(np.uint16), want)
    back = h_back.numpy()
    assert np.array_equal(back[dst_off:dst_off + host.nbytes].view(np.uint16), host)
    assert not back[:dst_off].any() and not back[dst_off + host.nbytes:].any()
