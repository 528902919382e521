"""swz_relayout_tma against the CPU oracle, bit-exact.

Where it applies, the relayout runs on the TMA's hardware swizzle modes
(swz_relayout_tma_path says which; the tests check it), so these tests also
pin the hardware: the 32-, 64- and 128-byte modes must produce exactly the
oracle's element Swizzle<B, 4 - log2(esize), 3>, B = 1, 2, 3, and the 128-byte
mode with 32-byte atoms the oracle's element Swizzle<2, 5 - log2(esize), 2>, in
both directions (each mode is its own inverse: both run as a swizzled tensor
load)."""
import numpy as np
import pytest

from gpu_util import empty_device, guards_intact, to_device, to_host, torch, void_dtype

pytestmark = pytest.mark.gpu

LOG2 = {1: 0, 2: 1, 4: 2, 8: 3, 16: 4}


@pytest.fixture(scope="module")
def swz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import xor_swizzle_movement_gb300 as m
    m.lib()
    return m


def run(swz, host, n_tiles, rows, cols, esize, B, M, S, direction, src_off=0, dst_off=0, path=None):
    nbytes = host.nbytes
    _, src = to_device(host, src_off)
    full, dst = empty_device(nbytes, dst_off)
    if path is not None:
        assert swz.swz_relayout_tma_path(dst, src, n_tiles, rows, cols, esize, B, M, S, direction) == path
    swz.swz_relayout_tma(dst, src, n_tiles, rows, cols, esize, B, M, S, direction)
    torch.cuda.synchronize()
    assert guards_intact(full, dst_off, nbytes)
    return to_host(dst, host.dtype)


@pytest.mark.parametrize("esize", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("B", [1, 2, 3])
@pytest.mark.parametrize("tile_bytes,n_tiles", [(1024, 37), (8192, 9), (3072, 11), (65536, 5)])
def test_hardware_modes(swz, orc, esize, B, tile_bytes, n_tiles):
    """Every element size and swizzle mode; tile counts that leave a partial
    last 8 KiB chunk; both directions."""
    from xor_swizzle_movement_gb300 import inputs
    M, S = 4 - LOG2[esize], 3
    tile = tile_bytes // esize
    cols = max(1, 128 // esize)
    rows = tile // cols
    host = inputs.random_bytes(n_tiles * tile_bytes, seed=11).view(void_dtype(esize))
    for direction in (0, 1):
        got = run(swz, host, n_tiles, rows, cols, esize, B, M, S, direction, path=B)
        want = orc.relayout(host, tile_elems=tile, B=B, M=M, S=S, direction=direction)
        assert got.tobytes() == want.tobytes(), direction
    assert swz.swz_device_status() == swz.SWZ_OK


@pytest.mark.parametrize("esize", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("tile_bytes,n_tiles", [(512, 37), (8192, 9), (1536, 11), (65536, 5)])
def test_atom32_mode(swz, orc, esize, tile_bytes, n_tiles):
    """The 128-byte mode with 32-byte atoms is element Swizzle<2, 5 - log2 e, 2>
    for every element size: 32-byte chunks XOR-ed with the 128-byte row mod 4."""
    from xor_swizzle_movement_gb300 import inputs
    B, M, S = 2, 5 - LOG2[esize], 2
    tile = tile_bytes // esize
    cols = max(1, 128 // esize)
    rows = tile // cols
    host = inputs.random_bytes(n_tiles * tile_bytes, seed=14).view(void_dtype(esize))
    for direction in (0, 1):
        got = run(swz, host, n_tiles, rows, cols, esize, B, M, S, direction, path=4)
        want = orc.relayout(host, tile_elems=tile, B=B, M=M, S=S, direction=direction)
        assert got.tobytes() == want.tobytes(), direction
    assert swz.swz_device_status() == swz.SWZ_OK


@pytest.mark.parametrize("B", [1, 2, 3])
@pytest.mark.parametrize("n_tiles", [1, 3])
def test_buffer_smaller_than_one_chunk(swz, orc, B, n_tiles):
    """Tiles of one swizzle period (2^(B+7) bytes) and a whole buffer below
    one 8 KiB chunk: the tensor box is taller than the tensor."""
    from xor_swizzle_movement_gb300 import inputs
    tile_bytes = 1 << (B + 7)
    cols = 64
    rows = tile_bytes // 2 // cols
    host = inputs.uint16_bits(n_tiles * tile_bytes // 2, seed=12)
    for direction in (0, 1):
        got = run(swz, host, n_tiles, rows, cols, 2, B, 3, 3, direction, path=B)
        want = orc.relayout(host, tile_elems=tile_bytes // 2, B=B, M=3, S=3, direction=direction)
        assert np.array_equal(got, want), direction
    assert swz.swz_device_status() == swz.SWZ_OK


def test_small_fp16_tiles_sw333(swz, orc):
    """256 tiles of 64 x 64 16-bit elements, Swizzle<3,3,3>: the 128-byte mode."""
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.uint16_bits(256 * 64 * 64, seed=0)
    for direction in (0, 1):
        got = run(swz, host, 256, 64, 64, 2, 3, 3, 3, direction)
        assert np.array_equal(got, orc.relayout(host, tile_elems=4096, B=3, M=3, S=3, direction=direction))


@pytest.mark.slow
def test_fp16_1gib_sw333(swz, orc):
    """One 1 GiB buffer of 16-bit elements in 64 x 64 tiles, forward and inverse,
    checked on 2^20 sampled positions and by the round trip."""
    n_tiles = (1 << 30) // 8192
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    src = torch.randint(0, 256, (1 << 30,), dtype=torch.uint8, device="cuda", generator=g)
    fwd = torch.empty_like(src)
    back = torch.empty_like(src)
    swz.swz_relayout_tma(fwd, src, n_tiles, 64, 64, 2, 3, 3, 3, 0)
    swz.swz_relayout_tma(back, fwd, n_tiles, 64, 64, 2, 3, 3, 3, 1)
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    rng = np.random.default_rng(2)
    idx = np.sort(rng.choice(n_tiles * 4096, 1 << 20, replace=False)).astype(np.int64)
    pos = orc.relayout_positions(idx, tile_elems=4096, B=3, M=3, S=3)
    assert torch.equal(fwd.view(torch.int16)[torch.from_numpy(pos).cuda()],
                       src.view(torch.int16)[torch.from_numpy(idx).cuda()])


@pytest.mark.parametrize("case", [
    dict(esize=2, rows=64, cols=64, B=3, M=4, S=3, n_tiles=4),     # not a hardware mode (M)
    dict(esize=2, rows=64, cols=64, B=3, M=3, S=2, n_tiles=4),     # not a hardware mode (S)
    dict(esize=2, rows=8, cols=32, B=3, M=3, S=3, n_tiles=7),      # 512-byte tiles < 1024-byte period
    dict(esize=4, rows=32, cols=32, B=5, M=0, S=5, n_tiles=3),     # B beyond the modes
    dict(esize=2, rows=2, cols=64, B=2, M=4, S=2, n_tiles=5),      # 256-byte tiles < the 32-byte-atom period
    dict(esize=2, rows=64, cols=64, B=1, M=5, S=1, n_tiles=3),     # 64-byte atoms: not routed
])
def test_fallback_matches_oracle(swz, orc, case):
    """Requests the TMA modes cannot express run the register kernels."""
    from xor_swizzle_movement_gb300 import inputs
    c = case
    tile = c["rows"] * c["cols"]
    host = inputs.random_bytes(c["n_tiles"] * tile * c["esize"], seed=12).view(void_dtype(c["esize"]))
    for direction in (0, 1):
        got = run(swz, host, c["n_tiles"], c["rows"], c["cols"], c["esize"], c["B"], c["M"], c["S"], direction,
                  path=0)
        want = orc.relayout(host, tile_elems=tile, B=c["B"], M=c["M"], S=c["S"], direction=direction)
        assert got.tobytes() == want.tobytes()


def test_misaligned_falls_back(swz, orc):
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.uint16_bits(16 * 64 * 64, seed=13)
    got = run(swz, host, 16, 64, 64, 2, 3, 3, 3, 0, src_off=2, dst_off=6, path=0)
    assert np.array_equal(got, orc.relayout(host, tile_elems=4096, B=3, M=3, S=3, direction=0))
