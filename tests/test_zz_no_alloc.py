"""The allocation-free TMA transpose against the regular one.

Some callers cannot let this library allocate device memory: their device
memory is planned ahead and owned by their own pool (a serving loop), or it
is already fully reserved by another allocator.  swz_transpose(...,
SWZ_T_TMA) makes one small cudaMalloc on its first call on a device;
swz_transpose_tma_noalloc serves those callers with a fixed array in the
library's device data instead.  These tests check, through the C ABI, that it
computes exactly what swz_transpose(..., SWZ_T_TMA) computes, on two calls in
a row (the second call reuses the array the first one left behind).

The file name sorts last, so a run that stops at the first failure has
already run every other test when it gets here.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import xor_swizzle_movement_gb300 as m
    m.lib()
    return m


def _matrix(rows, cols, seed):
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.f16_bits_no_nan(rows * cols, seed=seed).view(np.int16).reshape(rows, cols)
    return torch.from_numpy(host.copy()).cuda()


@pytest.mark.parametrize("rows,cols", [(1024, 2048), (200, 136), (96, 100)])
def test_noalloc_matches_tma_two_calls(swz, rows, cols):
    """(1024, 2048): whole TMA tiles; (200, 136): ragged edge tiles;
    (96, 100): cols not a multiple of 8, the shared-memory fallback."""
    for call, seed in enumerate((3, 11)):
        src = _matrix(rows, cols, seed)
        want = torch.empty(cols, rows, dtype=torch.int16, device="cuda")
        swz.swz_transpose(want, src, rows, cols, 2, swz.SWZ_T_TMA)
        got = torch.full((cols, rows), -1, dtype=torch.int16, device="cuda")
        if call == 0:
            assert swz.swz_transpose_tma_noalloc(got, src, rows, cols, wait=True) == 0
        else:
            assert swz.swz_transpose_tma_noalloc(got, src, rows, cols) == 0
            torch.cuda.synchronize()
        assert torch.equal(got, want), (rows, cols, call)


def test_noalloc_refuses_beyond_its_limit(swz):
    a = torch.zeros(64, dtype=torch.int16, device="cuda")
    b = torch.zeros(64, dtype=torch.int16, device="cuda")
    with pytest.raises(swz.SwzError) as e:
        swz.swz_transpose_tma_noalloc(b, a, 1 << 31, 8)
    assert e.value.status == swz.SWZ_ERR_SHAPE
    with pytest.raises(swz.SwzError) as e:
        swz.swz_transpose_tma_noalloc(a, a, 8, 8)
    assert e.value.status == swz.SWZ_ERR_ALIAS
