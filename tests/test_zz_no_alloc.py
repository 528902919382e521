"""The allocation-free TMA transpose against the oracle and the regular call.

Some callers cannot let this library allocate device memory: their device
memory is planned ahead and owned by their own pool (a serving loop), or it
is already fully reserved by another allocator.  swz_transpose(...,
SWZ_T_TMA) makes one small cudaMalloc on its first call on a device;
swz_transpose_tma_noalloc serves those callers with a fixed array in the
library's device data instead.  These tests check, through the C ABI, that it
computes the oracle's transpose and exactly what swz_transpose(...,
SWZ_T_TMA) computes, on two calls in a row (the second call reuses the array
the first one left behind), and that a bounded wait that gives up is reported
through that array.

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


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.lib()
    return oracle


def _host(rows, cols, seed):
    from xor_swizzle_movement_gb300 import inputs
    return inputs.f16_bits_no_nan(rows * cols, seed=seed).reshape(rows, cols)


def _bits(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("rows,cols", [(1024, 2048), (200, 136), (96, 100)])
def test_noalloc_matches_oracle_and_tma_two_calls(swz, orc, rows, cols):
    """(1024, 2048): whole TMA tiles; (200, 136): ragged edge tiles;
    (96, 100): cols not a multiple of 8, the shared-memory fallback."""
    for call, seed in enumerate((3, 11)):
        host = _host(rows, cols, seed)
        src = torch.from_numpy(host.view(np.int16).copy()).cuda()
        want = orc.transpose(host)
        regular = torch.empty(cols, rows, dtype=torch.int16, device="cuda")
        swz.swz_transpose(regular, src, rows, cols, 2, swz.SWZ_T_TMA)
        got = torch.full((cols, rows), -1, dtype=torch.int16, device="cuda")
        if call == 0:
            assert swz.swz_transpose_tma_noalloc(got, src, rows, cols, wait=True) == 0
        else:
            assert swz.swz_transpose_tma_noalloc(got, src, rows, cols) == 0
            torch.cuda.synchronize()
        assert np.array_equal(_bits(got), want), (rows, cols, call)
        assert torch.equal(got, regular), (rows, cols, call)


def test_noalloc_timeout_reported_through_its_array(swz, orc):
    """With no copy issued every bounded wait expires after 1 ms; the kernel
    records it in the fixed array's status word, the call reports it, dst is
    left untouched, and the next regular call (which clears the word first)
    reports no timeout and computes the transpose."""
    rows, cols = 256, 256
    host = _host(rows, cols, 5)
    src = torch.from_numpy(host.view(np.int16).copy()).cuda()
    dst = torch.full((cols, rows), 0x5A5A, dtype=torch.int16, device="cuda")
    flag, status = swz.swz_selftest_noalloc_timeout(dst, src, rows, cols, 1_000_000)
    assert (flag, status) == (1, swz.SWZ_ERR_TIMEOUT)
    assert bool((dst == 0x5A5A).all())
    assert swz.swz_transpose_tma_noalloc(dst, src, rows, cols, wait=True) == 0
    assert np.array_equal(_bits(dst), orc.transpose(host))


def test_noalloc_refuses_beyond_its_limit(swz):
    a = torch.zeros(64, dtype=torch.int16, device="cuda")
    b = torch.zeros(64, dtype=torch.int16, device="cuda")
    with pytest.raises(swz.SwzError) as e:
        swz.swz_transpose_tma_noalloc(b, a, 1 << 31, 8)
    assert e.value.status == swz.SWZ_ERR_SHAPE
    with pytest.raises(swz.SwzError) as e:
        swz.swz_transpose_tma_noalloc(a, a, 8, 8)
    assert e.value.status == swz.SWZ_ERR_ALIAS
