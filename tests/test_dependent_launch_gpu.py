"""Chains of launches that hand buffers back and forth with no host
synchronisation in between.  The kernels are launched with programmatic
dependent launch, so each may start before its predecessor finishes; every
launch below reads what the previous one wrote (read after write) and writes
what the previous one read (write after read).  The chains must end exactly
where the oracle says."""
import numpy as np
import pytest

from gpu_util import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import xor_swizzle_movement_gb300 as m
    m.lib()
    return m


def test_relayout_ping_pong(swz, orc):
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.bf16_normal(512 * 128 * 64, seed=1)
    a = torch.from_numpy(host.view(np.int16).copy()).cuda()
    b = torch.empty_like(a)
    for _ in range(50):
        swz.swz_relayout(b, a, 512, 128, 64, 2, 3, 4, 3, 0)   # a -> b forward
        swz.swz_relayout(a, b, 512, 128, 64, 2, 3, 4, 3, 1)   # b -> a inverse
    swz.swz_relayout(b, a, 512, 128, 64, 2, 3, 4, 3, 0)
    torch.cuda.synchronize()
    assert np.array_equal(a.cpu().numpy().view(np.uint16), host)
    want = orc.relayout(host, tile_elems=128 * 64, B=3, M=4, S=3, direction=0)
    assert np.array_equal(b.cpu().numpy().view(np.uint16), want)


def test_relayout_chain_s_less_than_b(swz, orc):
    """Swizzle<3,0,1> is not its own inverse: 7 forward steps in a row, then
    compare with the oracle applied 7 times."""
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.uint16_bits(64 * 1024, seed=0)
    bufs = [torch.from_numpy(host.view(np.int16).copy()).cuda(), torch.empty(64 * 1024, dtype=torch.int16, device="cuda")]
    want = host
    for i in range(7):
        swz.swz_relayout(bufs[(i + 1) % 2], bufs[i % 2], 64, 32, 32, 2, 3, 0, 1, 0)
        want = orc.relayout(want, tile_elems=1024, B=3, M=0, S=1, direction=0)
    torch.cuda.synchronize()
    assert np.array_equal(bufs[1].cpu().numpy().view(np.uint16), want)


@pytest.mark.parametrize("esize,n", [(4, 1024), (2, 2048), (8, 512), (1, 512)])
def test_transpose_ping_pong(swz, orc, esize, n):
    from xor_swizzle_movement_gb300 import inputs
    host = inputs.random_bytes(n * n * esize, seed=17)
    a = torch.from_numpy(host.copy()).cuda()
    b = torch.empty_like(a)
    for _ in range(20):
        swz.swz_transpose(b, a, n, n, esize, 0)
        swz.swz_transpose(a, b, n, n, esize, 0)
    swz.swz_transpose(b, a, n, n, esize, 0)
    torch.cuda.synchronize()
    assert np.array_equal(a.cpu().numpy(), host)
    dt = np.dtype(f"V{esize}")
    want = orc.transpose(host.view(dt).reshape(n, n))
    assert b.cpu().numpy().tobytes() == want.tobytes()


def test_mixed_kernels_chain(swz, orc):
    """Relayout, transpose, fused transpose-relayout and bank profiler launched
    back to back on one stream, each consuming the previous result."""
    from xor_swizzle_movement_gb300 import inputs
    n = 1024
    host = inputs.f16_bits_no_nan(n * n, seed=3)
    a = torch.from_numpy(host.view(np.int16).copy()).cuda()
    b, c, d = torch.empty_like(a), torch.empty_like(a), torch.empty_like(a)
    swz.swz_relayout(b, a, n * n // 4096, 64, 64, 2, 3, 3, 3, 0)      # b = relayout(a)
    swz.swz_transpose(c, b, n, n, 2, 0)                                # c = b^T
    swz.swz_transpose_relayout(d, c, n, n, 2, 4096, 3, 3, 3)          # d = relayout(c^T) = relayout(b)
    swz.swz_relayout(c, d, n * n // 4096, 64, 64, 2, 3, 3, 3, 1)      # c = inverse(d) = b
    torch.cuda.synchronize()
    want_b = orc.relayout(host, tile_elems=4096, B=3, M=3, S=3, direction=0)
    assert np.array_equal(b.cpu().numpy().view(np.uint16), want_b)
    assert np.array_equal(c.cpu().numpy().view(np.uint16), want_b)
