"""The largest parameters and sizes: Swizzle<16,0,16> across one 4 GiB tile
(offsets past 2^31 and 2^32 bytes), and a 65536 x 65536 fp16 transpose
(2^32 elements, 8 GiB), checked on samples the oracle computes."""
import numpy as np
import pytest

from gpu_util import torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def swz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import xor_swizzle_movement_gb300 as m
    m.lib()
    return m


def test_relayout_b16_one_4gib_tile(swz, orc):
    n = 1 << 32                          # uint8 elements in one tile
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    src = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)
    fwd = torch.empty_like(src)
    swz.swz_relayout(fwd, src, 1, 1 << 16, 1 << 16, 1, 16, 0, 16, 0)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    idx = np.concatenate([rng.integers(0, n, 1 << 18), [0, n - 1, (1 << 31) - 1, 1 << 31, (1 << 32) - 17]])
    idx = np.unique(idx).astype(np.int64)
    pos = orc.relayout_positions(idx, tile_elems=n, B=16, M=0, S=16)
    assert torch.equal(fwd[torch.from_numpy(pos).cuda()], src[torch.from_numpy(idx).cuda()])
    back = src  # reuse: the inverse overwrites src's storage only after the check above
    ref = src.clone()
    swz.swz_relayout(back, fwd, 1, 1 << 16, 1 << 16, 1, 16, 0, 16, 1)
    torch.cuda.synchronize()
    assert torch.equal(back, ref)


@pytest.mark.parametrize("variant", [0, 3])
def test_transpose_2pow32_fp16(swz, orc, variant):
    n = 1 << 16
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    src = torch.randint(-32768, 32768, (n, n), dtype=torch.int16, device="cuda", generator=g)
    dst = torch.empty_like(src)
    swz.swz_transpose(dst, src, n, n, 2, variant)
    torch.cuda.synchronize()
    rng = np.random.default_rng(6)
    corners = [(0, 0), (n - 32, n - 32), (0, n - 32), (n - 32, 0)]
    corners += [tuple(int(v) for v in rng.integers(0, n - 32, 2)) for _ in range(60)]
    for r0, c0 in corners:
        block = src[r0:r0 + 32, c0:c0 + 32].cpu().numpy()
        want = orc.transpose(block)
        got = dst[c0:c0 + 32, r0:r0 + 32].cpu().numpy()
        assert np.array_equal(got, want), (r0, c0)
