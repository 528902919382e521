"""GPU bank profiler and batched slice collision against the CPU oracle
(exact integer results)."""
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


def gpu_profile(swz, pats, width, active=None):
    n = pats.shape[0]
    dp = torch.from_numpy(np.ascontiguousarray(pats, dtype=np.uint32).view(np.int32)).cuda()
    da = None if active is None else torch.from_numpy(active.view(np.int32)).cuda()
    w = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    f = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    swz.swz_bank_profile(dp, da, n, width, w, f)
    torch.cuda.synchronize()
    return w.cpu().numpy(), f.cpu().numpy()


def structured_patterns():
    """Column/row/broadcast/swizzled patterns of the oracle pins, as rows of 32 addresses."""
    pats = []
    for col in range(32):
        pats.append([4 * (r * 32 + col) for r in range(32)])            # fp32 column
        pats.append([4 * (r * 33 + col) for r in range(32)])            # padded
        pats.append([4 * (r * 32 + (col ^ r)) for r in range(32)])      # XOR swizzle
    pats.append([4 * c for c in range(32)])                             # row
    pats.append([128] * 32)                                             # broadcast
    pats.append([(l % 2) * 2 for l in range(32)])                       # halves of one word
    pats.append([16 * l for l in range(32)])                            # 512 contiguous bytes
    return np.array(pats, dtype=np.uint32)


@pytest.mark.parametrize("width", [1, 2, 4, 8, 16])
def test_structured(swz, orc, width):
    pats = structured_patterns()
    pats = (pats // width) * width  # aligned to the access width
    gw, gf = gpu_profile(swz, pats, width)
    ow, of = orc.bank_profile(pats, width)
    assert np.array_equal(gw, ow) and np.array_equal(gf, of)


@pytest.mark.parametrize("width", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("aligned", [True, False])
@pytest.mark.parametrize("masked", [False, True])
def test_random(swz, orc, width, aligned, masked):
    from xor_swizzle_movement_gb300 import inputs
    n = 8192
    pats = inputs.bank_patterns(n, width, seed=5, aligned=aligned)
    # narrow address ranges force collisions and shared words
    pats[: n // 2] %= 512
    act = inputs.active_masks(n, seed=6) if masked else None
    if masked:
        act[:16] = 0
    gw, gf = gpu_profile(swz, pats, width, act)
    ow, of = orc.bank_profile(pats, width, act)
    assert np.array_equal(gw, ow) and np.array_equal(gf, of)


def gpu_profile_offset(swz, pats, width, active=None, word_offset=1):
    """As gpu_profile, with the address and mask arrays starting word_offset
    words into their buffers (off 16-byte alignment for odd offsets)."""
    n = pats.shape[0]
    flat = np.zeros(n * 32 + word_offset, dtype=np.uint32)
    flat[word_offset:] = pats.reshape(-1)
    dp = torch.from_numpy(flat.view(np.int32)).cuda()[word_offset:]
    da = None
    if active is not None:
        fa = np.zeros(n + word_offset, dtype=np.uint32)
        fa[word_offset:] = active
        da = torch.from_numpy(fa.view(np.int32)).cuda()[word_offset:]
    w = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    f = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    swz.swz_bank_profile(dp, da, n, width, w, f)
    torch.cuda.synchronize()
    return w.cpu().numpy(), f.cpu().numpy()


def mixed_patterns(n, width, seed):
    """Aligned random patterns, every third one with some lanes moved off
    alignment, some squeezed into 512 bytes (shared words, deep conflicts) and
    some near the top of the 32-bit address space."""
    rng = np.random.default_rng(seed)
    pats = (rng.integers(0, 228 * 1024 // width, (n, 32)) * width).astype(np.uint64)
    pats[1::5] %= 512
    pats[2::7] += (1 << 32) - 228 * 1024
    bad = np.arange(n) % 3 == 0
    shift = rng.integers(0, 2, (n, 32)) * rng.integers(1, 16, (n, 32))
    pats[bad] += shift[bad].astype(np.uint64)
    return (pats % (1 << 32)).astype(np.uint32)


@pytest.mark.parametrize("width", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("n", [1, 31, 33, 97, 4099])
@pytest.mark.parametrize("masked", [False, True])
def test_ragged_mixed(swz, orc, width, n, masked):
    """Pattern counts that leave a partial batch of 32, aligned and unaligned
    patterns side by side in one batch (the unaligned ones take the exact
    count), masks that switch off whole passes or only the unaligned lanes."""
    pats = mixed_patterns(n, width, seed=n + width)
    act = None
    if masked:
        act = inputs_masks(n, seed=n)
        act[::4] = 0xFFFF0000
        act[1::4] = 0x000000FF
        act[2::9] = 0
        # switch off exactly the unaligned lanes of some patterns: they count as aligned
        for p in range(0, n, 6):
            off = (pats[p] % max(width, 1)) != 0 if width > 4 else ((pats[p] & 3) + width > 4)
            act[p] = np.uint32(sum(1 << l for l in range(32) if not off[l]))
    gw, gf = gpu_profile(swz, pats, width, act)
    ow, of = orc.bank_profile(pats, width, act)
    assert np.array_equal(gw, ow) and np.array_equal(gf, of)


@pytest.mark.parametrize("width", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("masked", [False, True])
def test_address_array_off_16_bytes(swz, orc, width, masked):
    """Address and mask arrays 4 and 12 bytes past a 16-byte boundary: the
    patterns are staged word by word instead of in 16-byte chunks."""
    n = 1000
    pats = mixed_patterns(n, width, seed=40 + width)
    act = inputs_masks(n, seed=41) if masked else None
    ow, of = orc.bank_profile(pats, width, act)
    for off in (1, 3):
        gw, gf = gpu_profile_offset(swz, pats, width, act, word_offset=off)
        assert np.array_equal(gw, ow) and np.array_equal(gf, of)


@pytest.mark.parametrize("width", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("masked", [False, True])
def test_key_range_edges(swz, orc, width, masked):
    """Addresses around 2^18 - 16 bytes (where 16-bit keys give way to 32-bit
    ones) and at the top of the 32-bit space (an access's last word past
    2^30 - 1), aligned and unaligned, each edge alone in its batches and
    mixed with small addresses."""
    rng = np.random.default_rng(60 + width)
    n = 64 * 12
    pats = rng.integers(0, 4096, (n, 32)).astype(np.int64) * 4
    edges = [(1 << 18) - 40, (1 << 18) - 17, (1 << 18) - 16, (1 << 18) - 4, (1 << 32) - 64, (1 << 32) - 16]
    for b, e in enumerate(edges):
        blk = slice(64 * 2 * b, 64 * 2 * b + 64)      # the edge in a whole batch
        pats[blk] = e + rng.integers(0, 40, (64, 32))
        pats[64 * 2 * b + 64 + 5] = e + rng.integers(0, 40, 32)  # one row in a batch of small ones
    pats = np.minimum(pats, (1 << 32) - 1)
    aligned = rng.random(n) < 0.5
    pats[aligned] = pats[aligned] // width * width
    pats = pats.astype(np.uint32)
    act = None
    if masked:
        act = inputs_masks(n, seed=61)
        act[::5] = 0x80000001
    gw, gf = gpu_profile(swz, pats, width, act)
    ow, of = orc.bank_profile(pats, width, act)
    assert np.array_equal(gw, ow) and np.array_equal(gf, of)


def inputs_masks(n, seed):
    from xor_swizzle_movement_gb300 import inputs
    return inputs.active_masks(n, seed=seed)


@pytest.mark.slow
def test_bench_size(swz, orc):
    """2^22 aligned random 4-byte patterns: the benchmark's profiler batch."""
    from xor_swizzle_movement_gb300 import inputs
    n = 1 << 22
    pats = inputs.bank_patterns(n, 4, seed=5)
    gw, gf = gpu_profile(swz, pats, 4)
    ow, of = orc.bank_profile(pats, 4)
    assert np.array_equal(gw, ow) and np.array_equal(gf, of)


@pytest.mark.slow
@pytest.mark.parametrize("width,masked,unaligned", [(1, False, False), (2, False, False), (8, False, False),
                                                   (16, False, False), (4, True, False), (4, False, True),
                                                   (16, True, True)])
def test_bench_size_other_widths(swz, orc, width, masked, unaligned):
    """2^22 random patterns, as the benchmark's other profiler rows: every
    access width, lane masks, and patterns moved 2 bytes off alignment (the
    word-key count)."""
    from xor_swizzle_movement_gb300 import inputs
    n = 1 << 22
    pats = inputs.bank_patterns(n, width, seed=5)
    if unaligned:
        pats += 2
    act = inputs.active_masks(n, seed=6) if masked else None
    gw, gf = gpu_profile(swz, pats, width, act)
    ow, of = orc.bank_profile(pats, width, act)
    assert np.array_equal(gw, ow) and np.array_equal(gf, of)


def test_errors(swz):
    w = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(swz.SwzError) as e:
        swz.swz_bank_profile(w, None, 1, 3, w, w)
    assert e.value.status == swz.SWZ_ERR_PARAM
    with pytest.raises(swz.SwzError) as e:
        swz.swz_bank_profile(None, None, 1, 4, w, w)
    assert e.value.status == swz.SWZ_ERR_NULL
    swz.swz_bank_profile(None, None, 0, 4, None, None)  # empty


@pytest.mark.parametrize("B,M,S", [(3, 2, 4), (3, 3, 3), (2, 0, 1), (5, 0, 5), (4, 4, 11)])
def test_slice_collision_batch(swz, orc, B, M, S):
    masks = np.concatenate([np.arange(1 << 16, dtype=np.uint64),
                            np.random.default_rng(3).integers(0, 2**63, 4096, dtype=np.uint64)])
    dA = torch.from_numpy(masks.view(np.int64)).cuda()
    dC = torch.empty_like(dA)
    swz.swz_slice_collision_batch(dA, masks.size, B, M, S, dC)
    torch.cuda.synchronize()
    got = dC.cpu().numpy().view(np.uint64)
    want = np.array([orc.slice_collision(int(a), B=B, M=M, S=S) for a in masks], dtype=np.uint64)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("n,a_off,c_off,in_place", [
    (1001, 0, 0, False),   # odd count: pairs by 16-byte accesses, the last mask on its own
    (1000, 8, 0, False),   # masks off 16-byte alignment: element by element
    (999, 0, 8, False),
    (4097, 0, 0, True),    # in place (A == C)
    (1, 0, 0, False),
])
def test_slice_collision_batch_shapes(swz, orc, n, a_off, c_off, in_place):
    B, M, S = 3, 1, 2
    masks = np.random.default_rng(n).integers(0, 2**63, n, dtype=np.uint64)
    bufA = torch.zeros(n + 2, dtype=torch.int64, device="cuda")
    bufA.view(torch.uint8)[a_off:a_off + 8 * n].copy_(torch.from_numpy(masks.view(np.uint8)).cuda())
    pa = bufA.data_ptr() + a_off
    bufC = bufA if in_place else torch.full((n + 2,), -1, dtype=torch.int64, device="cuda")
    pc = pa if in_place else bufC.data_ptr() + c_off
    swz.swz_slice_collision_batch(pa, n, B, M, S, pc)
    torch.cuda.synchronize()
    raw = bufC.view(torch.uint8).cpu().numpy()
    off = a_off if in_place else c_off
    got = raw[off:off + 8 * n].view(np.uint64)
    want = np.array([orc.slice_collision(int(a), B=B, M=M, S=S) for a in masks], dtype=np.uint64)
    assert np.array_equal(got, want)
    if not in_place:  # nothing written outside the n masks
        assert (raw[:off] == 0xFF).all() and (raw[off + 8 * n:] == 0xFF).all()
