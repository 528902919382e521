"""swz_transpose_relayout (transpose fused with a forward relayout) against
the CPU oracle's two steps, bit-exact."""
import numpy as np
import pytest

from gpu_util import empty_device, guards_intact, to_device, to_host, torch, void_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import xor_swizzle_movement_gb300 as m
    m.lib()
    return m


def run(swz, host, esize, te, B, M, S, src_off=0, dst_off=0):
    rows, cols = host.shape
    nbytes = host.nbytes
    _, src = to_device(host, src_off)
    full, dst = empty_device(nbytes, dst_off)
    swz.swz_transpose_relayout(dst, src, rows, cols, esize, te, B, M, S)
    torch.cuda.synchronize()
    assert guards_intact(full, dst_off, nbytes)
    return to_host(dst, host.dtype)


BMS = [(3, 4, 3), (3, 3, 3), (5, 0, 5), (2, 1, 3), (3, 0, 1), (4, 1, 2), (0, 0, 3), (5, 2, 5)]
SHAPES = [(64, 128), (128, 64), (96, 160), (200, 136), (48, 256)]


def tile_for(rows, cols, B, M):
    """Relayout tiles of whole rows of the transposed matrix where they close
    under the swizzle, else the smallest closed multiple that divides the
    matrix; None when the matrix cannot be cut into closed tiles that way."""
    n = rows * cols
    for k in (8, 4, 2, 1, 16, 32, 64):
        cand = k * rows
        if n % cand == 0 and cand % (1 << (M + B)) == 0:
            return cand
    return None


# only the (swizzle, shape) pairs whose matrix splits into closed tiles
CASES = [(bms, shape) for bms in BMS for shape in SHAPES if tile_for(*shape, bms[0], bms[1]) is not None]


@pytest.mark.parametrize("esize", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("bms,shape", CASES)
def test_matches_oracle(swz, orc, esize, bms, shape):
    from xor_swizzle_movement_gb300 import inputs
    B, M, S = bms
    rows, cols = shape
    n = rows * cols
    te = tile_for(rows, cols, B, M)
    host = inputs.random_bytes(n * esize, seed=14).view(void_dtype(esize)).reshape(rows, cols)
    got = run(swz, host, esize, te, B, M, S)
    want = orc.transpose_relayout(host, tile_elems=te, B=B, M=M, S=S)
    assert got.tobytes() == want.tobytes()


@pytest.mark.parametrize("te", [64 * 24, 64 * 40, 64 * 8])
def test_tile_local_offsets(swz, orc, te):
    """Tiles that do not hold a multiple of the swizzle period (512 elements
    for Swizzle<3,3,3>): offsets are tile-local."""
    from xor_swizzle_movement_gb300 import inputs
    rows, cols = 64, 480
    host = inputs.f16_bits_no_nan(rows * cols, seed=15).reshape(rows, cols)
    got = run(swz, host, 2, te, 3, 3, 3)
    assert np.array_equal(got, orc.transpose_relayout(host, tile_elems=te, B=3, M=3, S=3))


def test_k_major_operand_tiles(swz, orc):
    """A 64 x 65536 bf16 matrix becomes 512 K-major 128 x 64 tiles under
    Swizzle<3,4,3> (the tile of the headline relayout) in one pass."""
    from xor_swizzle_movement_gb300 import inputs
    rows, cols = 64, 65536
    host = inputs.bf16_normal(rows * cols, seed=1).reshape(rows, cols)
    got = run(swz, host, 2, 128 * 64, 3, 4, 3)
    assert np.array_equal(got, orc.transpose_relayout(host, tile_elems=128 * 64, B=3, M=4, S=3))
    # the same result as the two steps on the GPU
    src = torch.from_numpy(host.view(np.int16).copy()).cuda()
    t = torch.empty(cols * rows, dtype=torch.int16, device="cuda")
    two = torch.empty_like(t)
    swz.swz_transpose(t, src, rows, cols, 2, swz.SWZ_T_SWIZZLED)
    swz.swz_relayout(two, t, cols * rows // 8192, 128, 64, 2, 3, 4, 3, 0)
    torch.cuda.synchronize()
    assert np.array_equal(two.cpu().numpy().view(np.uint16), got)


@pytest.mark.parametrize("esize", [1, 2, 4, 8, 16])
def test_misaligned(swz, orc, esize):
    from xor_swizzle_movement_gb300 import inputs
    rows, cols = 64, 128
    host = inputs.random_bytes(rows * cols * esize, seed=16).view(void_dtype(esize)).reshape(rows, cols)
    got = run(swz, host, esize, 8 * rows, 3, 0, 3, src_off=esize, dst_off=3 * esize)
    assert got.tobytes() == orc.transpose_relayout(host, tile_elems=8 * rows, B=3, M=0, S=3).tobytes()


def test_errors(swz):
    a = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    b = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    for args, status in [((b, a, 16, 16, 4, 0, 3, 0, 3), swz.SWZ_ERR_SHAPE),      # tile_elems 0
                         ((b, a, 16, 16, 4, 96, 3, 0, 3), swz.SWZ_ERR_SHAPE),     # 96 does not divide 256
                         ((b, a, 16, 16, 4, 4, 3, 0, 3), swz.SWZ_ERR_SHAPE),      # 4 not closed under 2^3
                         ((b, a, 16, 16, 4, 64, 3, 0, 0), swz.SWZ_ERR_PARAM),
                         ((b, a, 16, 16, 3, 64, 3, 0, 3), swz.SWZ_ERR_PARAM),
                         ((a, a, 16, 16, 4, 64, 3, 0, 3), swz.SWZ_ERR_ALIAS)]:
        with pytest.raises(swz.SwzError) as e:
            swz.swz_transpose_relayout(*args)
        assert e.value.status == status, args
