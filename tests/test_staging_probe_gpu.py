"""The shared-memory staging probe (swz_staging_probe through the C ABI).

The probe repeats a transpose staging's fill and drain on register data; it
exists so that the hardware bank-conflict counters can be read on the staging
alone.  Each staging maps a tile element (row, col) to a shared address one
to one, and the fill and the drain use the same map, so what a thread reads
back does not depend on the layout: the swizzled, unswizzled and padded
stagings of one element size must give the same per-CTA checksums, with and
without the streamed global traffic."""
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


def _sums(swz, esize, variant, ctas, iters, g=None):
    sink = torch.zeros(ctas, dtype=torch.int32, device="cuda")
    if g is None:
        swz.swz_staging_probe(esize, variant, iters, ctas, sink=sink)
    else:
        swz.swz_staging_probe(esize, variant, iters, ctas, gsrc=g[0], gdst=g[1], gbytes=g[0].numel(), sink=sink)
    torch.cuda.synchronize()
    return sink.cpu().numpy()


@pytest.mark.parametrize("esize", [2, 4, 8])
@pytest.mark.parametrize("with_global", [False, True])
def test_layouts_read_back_the_same(swz, esize, with_global):
    ctas, iters = 40, 5
    g = None
    if with_global:
        gen = torch.Generator(device="cuda")
        gen.manual_seed(7)
        src = torch.randint(0, 256, (1 << 20,), dtype=torch.uint8, device="cuda", generator=gen)
        g = (src, torch.empty_like(src))
    variants = [swz.SWZ_T_SWIZZLED, swz.SWZ_T_UNSWIZZLED, swz.SWZ_T_PADDED]
    if esize == 2:
        variants.append(swz.SWZ_T_TMA)   # the TMA kernel's staging: an stmatrix output tile as well
    sums = [_sums(swz, esize, v, ctas, iters, g) for v in variants]
    assert all(np.array_equal(sums[0], s) for s in sums[1:])
    # the CTAs differ only through the streamed data
    assert (len(set(sums[0].tolist())) > 1) == with_global
    if with_global:
        # every drain vector was stored: the destination is no longer the untouched allocation
        assert not torch.equal(g[1], torch.empty_like(g[1]).zero_())


def test_byte_staging_runs_and_rejects(swz):
    s = _sums(swz, 1, swz.SWZ_T_SWIZZLED, 16, 3)
    assert s.shape == (16,)
    with pytest.raises(swz.SwzError) as e:
        swz.swz_staging_probe(1, swz.SWZ_T_UNSWIZZLED, 1, 1)
    assert e.value.status == swz.SWZ_ERR_PARAM
    with pytest.raises(swz.SwzError) as e:
        swz.swz_staging_probe(4, swz.SWZ_T_TMA, 1, 1)
    assert e.value.status == swz.SWZ_ERR_PARAM
    with pytest.raises(swz.SwzError) as e:
        swz.swz_staging_probe(16, swz.SWZ_T_SWIZZLED, 1, 1)
    assert e.value.status == swz.SWZ_ERR_PARAM
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(swz.SwzError) as e:
        swz.swz_staging_probe(4, swz.SWZ_T_SWIZZLED, 1, 1, gsrc=buf, gdst=buf, gbytes=64)
    assert e.value.status == swz.SWZ_ERR_ALIAS
