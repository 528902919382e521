"""GPU transpose (swz_transpose through the C ABI) against the CPU oracle,
bit-exact, every element size and staging variant, tile-aligned and ragged
shapes, misaligned pointers, and the full-size fp32 / fp16 / fp64 matrices."""
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


VARIANTS = [0, 1, 2]
SHAPES = [(64, 64), (128, 192), (1, 1), (1, 100), (100, 1), (67, 45), (200, 136), (64, 72),
          (130, 66), (96, 520), (33, 257)]


def run_transpose(swz, host, esize, variant, src_off=0, dst_off=0):
    rows, cols = host.shape
    nbytes = host.nbytes
    _, src = to_device(host, src_off)
    full, dst = empty_device(nbytes, dst_off)
    swz.swz_transpose(dst, src, rows, cols, esize, variant)
    torch.cuda.synchronize()
    assert guards_intact(full, dst_off, nbytes)
    return to_host(dst, host.dtype, (cols, rows))


@pytest.mark.parametrize("esize", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SHAPES)
def test_shapes(swz, orc, esize, variant, shape):
    from xor_swizzle_movement_gb300 import inputs
    rows, cols = shape
    host = inputs.random_bytes(rows * cols * esize, seed=9).view(void_dtype(esize)).reshape(rows, cols)
    got = run_transpose(swz, host, esize, variant)
    assert got.tobytes() == orc.transpose(host).tobytes()


@pytest.mark.parametrize("esize", [2, 4, 8])
def test_misaligned(swz, orc, esize):
    from xor_swizzle_movement_gb300 import inputs
    rows, cols = 128, 128
    host = inputs.random_bytes(rows * cols * esize, seed=10).view(void_dtype(esize)).reshape(rows, cols)
    got = run_transpose(swz, host, esize, 0, src_off=esize, dst_off=2 * esize)
    assert got.tobytes() == orc.transpose(host).tobytes()


@pytest.mark.slow
@pytest.mark.parametrize("shape", [(2048, 4096), (384, 640), (4096, 2048 + 16)])
def test_u8_full_tiles(swz, orc, shape):
    """1-byte elements through 128 x 128 byte tiles: whole tiles (register 4 x 4
    byte transposes), and a column count that leaves a ragged last tile."""
    from xor_swizzle_movement_gb300 import inputs
    rows, cols = shape
    host = inputs.random_bytes(rows * cols, seed=17).reshape(rows, cols)
    for variant in VARIANTS:
        got = run_transpose(swz, host, 1, variant)
        assert np.array_equal(got, orc.transpose(host)), variant


def test_fp32_8192_all_variants(swz, orc):
    from xor_swizzle_movement_gb300 import inputs
    n = 8192
    host = inputs.f32_uniform(n * n, seed=2).reshape(n, n)
    want = orc.transpose(host).view(np.uint32)
    _, src = to_device(host)
    for variant in VARIANTS:
        full, dst = empty_device(host.nbytes)
        swz.swz_transpose(dst, src, n, n, 4, variant)
        torch.cuda.synchronize()
        assert guards_intact(full, 0, host.nbytes)
        assert np.array_equal(to_host(dst, np.uint32, (n, n)), want), variant


@pytest.mark.slow
def test_fp16_16384(swz, orc):
    from xor_swizzle_movement_gb300 import inputs
    n = 16384
    host = inputs.f16_bits_no_nan(n * n, seed=3).reshape(n, n)
    want = orc.transpose(host)
    _, src = to_device(host)
    for variant in (0, 3, 1, 2):   # swizzled, TMA, unswizzled, padded: every staging at full size
        full, dst = empty_device(host.nbytes)
        swz.swz_transpose(dst, src, n, n, 2, variant)
        torch.cuda.synchronize()
        assert guards_intact(full, 0, host.nbytes)
        assert np.array_equal(to_host(dst, np.uint16, (n, n)), want), variant
        del full, dst


@pytest.mark.slow
def test_fp64_8192(swz, orc):
    from xor_swizzle_movement_gb300 import inputs
    n = 8192
    host = inputs.random_bytes(n * n * 8, seed=4).view(np.uint64).reshape(n, n)
    want = orc.transpose(host)
    for variant in (0, 1, 2):      # swizzled, unswizzled, padded: every staging at full size
        got = run_transpose(swz, host, 8, variant)
        assert np.array_equal(got, want), variant
        del got


def test_errors(swz):
    _, a = empty_device(4096)
    _, b = empty_device(4096)
    swz.swz_transpose(b, a, 0, 16, 4, 0)  # empty: nothing launched
    for args, status in [((b, a, 16, 16, 3, 0), swz.SWZ_ERR_PARAM),
                         ((b, a, 16, 16, 4, 7), swz.SWZ_ERR_PARAM),
                         ((b, a, 16, 16, 4, 3), swz.SWZ_ERR_PARAM),   # TMA staging is 16-bit only
                         ((b, a, -1, 16, 4, 0), swz.SWZ_ERR_SHAPE),
                         ((a, a, 16, 16, 4, 0), swz.SWZ_ERR_ALIAS),
                         ((b[2:], a, 16, 16, 4, 0), swz.SWZ_ERR_ALIGN)]:
        with pytest.raises(swz.SwzError) as e:
            swz.swz_transpose(*args)
        assert e.value.status == status, args


# ---------------------------------------------------------------- TMA path --

@pytest.mark.parametrize("shape", [(64, 64), (128, 256), (200, 136), (100, 60), (1000, 1000), (8, 8),
                                   (64, 4096), (4096, 64), (130, 72)])
def test_tma_shapes(swz, orc, shape):
    from xor_swizzle_movement_gb300 import inputs
    rows, cols = shape
    host = inputs.f16_bits_no_nan(rows * cols, seed=3).reshape(rows, cols)
    got = run_transpose(swz, host, 2, swz.SWZ_T_TMA)
    assert np.array_equal(got, orc.transpose(host))
    assert swz.swz_device_status() == swz.SWZ_OK


def test_tma_bounded_wait_reports_timeout(swz, orc):
    """The TMA kernel's barrier waits give up after their limit: with no copy
    issued every wait expires, the kernel records SWZ_ERR_TIMEOUT and
    returns, the status reads back once, and the context stays usable."""
    from xor_swizzle_movement_gb300 import inputs
    rows, cols = 256, 256
    host = inputs.f16_bits_no_nan(rows * cols, seed=3).reshape(rows, cols)
    _, src = to_device(host)
    full, dst = empty_device(host.nbytes)
    assert swz.swz_device_status() == swz.SWZ_OK
    swz.swz_selftest_tma_timeout(dst, src, rows, cols, 1_000_000)
    assert swz.swz_device_status() == swz.SWZ_ERR_TIMEOUT
    assert swz.swz_device_status() == swz.SWZ_OK        # read clears it
    assert guards_intact(full, 0, host.nbytes)
    assert (dst.cpu().numpy() == 0xA5).all()             # nothing written
    swz.swz_transpose(dst, src, rows, cols, 2, swz.SWZ_T_TMA)
    assert swz.swz_device_status() == swz.SWZ_OK
    assert np.array_equal(to_host(dst, np.uint16, (cols, rows)), orc.transpose(host))
