"""Relayouts of a 64 GiB buffer: vector indices beyond 2^32 (and element
offsets beyond 2^35), where any 32-bit index arithmetic in a kernel or a
launcher would wrap.  Each path is checked at 2^16 random positions spread
over the whole buffer against the oracle's map, and forward then inverse must
give the input back everywhere (the input is regenerated chunk by chunk from
its seeds to compare)."""
import numpy as np
import pytest

from gpu_util import torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

GIB = 1 << 30
N_BYTES = 64 * GIB
CHUNK = GIB


@pytest.fixture(scope="module")
def swz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import xor_swizzle_movement_gb300 as m
    m.lib()
    return m


def _fill(buf):
    """Chunk i of the buffer: random bytes from seed 100 + i."""
    g = torch.Generator(device="cuda")
    for i in range(N_BYTES // CHUNK):
        g.manual_seed(100 + i)
        buf[i * CHUNK:(i + 1) * CHUNK].random_(0, 256, generator=g)


def _equal_to_input(buf):
    g = torch.Generator(device="cuda")
    want = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    for i in range(N_BYTES // CHUNK):
        g.manual_seed(100 + i)
        want.random_(0, 256, generator=g)
        if not torch.equal(buf[i * CHUNK:(i + 1) * CHUNK], want):
            return False
    return True


@pytest.fixture(scope="module")
def big():
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    if free < 170 * GIB:
        pytest.skip("needs 160 GiB of free device memory (two 64 GiB buffers and a 32 GiB copy)")
    src = torch.empty(N_BYTES, dtype=torch.uint8, device="cuda")
    dst = torch.empty(N_BYTES, dtype=torch.uint8, device="cuda")
    yield src, dst
    del src, dst
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,M,S", [(3, 3, 3),     # whole vectors, lanes XOR-ed in registers
                                   (3, 0, -4),    # negative shift: warp shuffles
                                   (4, 2, -9),    # negative shift: register cosets, 8 per thread
                                   (3, 0, -2)])   # negative shift: warp shuffles after a lane map
def test_relayout_64gib(swz, orc, big, B, M, S):
    src, dst = big
    n = N_BYTES // 2                              # uint16 elements, one tile
    _fill(src)
    rng = np.random.default_rng(B * 100 + M * 10 + S)
    idx = np.sort(rng.choice(n, 1 << 16, replace=False)).astype(np.int64)
    idx[-1] = n - 1                               # the last element
    ti = torch.from_numpy(idx).cuda()
    vals = src.view(torch.int16)[ti].clone()
    swz.swz_relayout(dst, src, 1, 1, n, 2, B, M, S, 0)
    torch.cuda.synchronize()
    pos = orc.relayout_positions(idx, tile_elems=n, B=B, M=M, S=S)
    assert torch.equal(dst.view(torch.int16)[torch.from_numpy(pos).cuda()], vals)
    swz.swz_relayout(src, dst, 1, 1, n, 2, B, M, S, 1)
    torch.cuda.synchronize()
    assert _equal_to_input(src)


@pytest.mark.parametrize("esize,variant", [(4, 0), (2, 0), (2, 3), (8, 0), (1, 0), (16, 0)])
def test_transpose_64gib(swz, big, esize, variant):
    """A 64 GiB matrix of 131072 rows (element offsets past 2^32; for the TMA
    variant, tensor maps of 131072 x 262144 elements), transposed on each
    element size's swizzled staging; 2^16 sampled elements checked, the last
    one included."""
    src, dst = big
    R = 131072
    C = N_BYTES // esize // R
    dt = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64, 16: torch.int64}[esize]
    w = esize // 8 if esize == 16 else 1          # 16-byte elements: two int64 words each
    swz.swz_transpose(dst, src, R, C, esize, variant)
    torch.cuda.synchronize()
    rng = np.random.default_rng(esize * 10 + variant)
    r = rng.integers(0, R, 1 << 16).astype(np.int64)
    c = rng.integers(0, C, 1 << 16).astype(np.int64)
    r[-1], c[-1] = R - 1, C - 1
    sv, dv = src.view(dt), dst.view(dt)
    for k in range(w):
        si = torch.from_numpy((r * C + c) * w + k).cuda()
        di = torch.from_numpy((c * R + r) * w + k).cuda()
        assert torch.equal(dv[di], sv[si])


def _check_relayout(swz, orc, fn, src, dst, n_tiles, tile, esize, B, M, S, seed):
    """dst = forward relayout of src (views of the big buffers), checked at
    2^16 sampled elements (the last one included) against the oracle's map,
    then inverse back into src and compared with the saved input."""
    dt = {1: torch.uint8, 2: torch.int16}[esize]
    n = n_tiles * tile
    keep = src.clone() if src.numel() < N_BYTES else None
    rng = np.random.default_rng(seed)
    idx = np.sort(rng.choice(n, 1 << 16, replace=False)).astype(np.int64)
    idx[-1] = n - 1
    ti = torch.from_numpy(idx).cuda()
    vals = src.view(dt)[ti].clone()
    fn(dst, src, n_tiles, 1, tile, esize, B, M, S, 0)
    torch.cuda.synchronize()
    pos = orc.relayout_positions(idx, tile_elems=tile, B=B, M=M, S=S)
    assert torch.equal(dst.view(dt)[torch.from_numpy(pos).cuda()], vals)
    fn(src, dst, n_tiles, 1, tile, esize, B, M, S, 1)
    torch.cuda.synchronize()
    if keep is not None:
        assert torch.equal(src, keep)
    else:
        assert _equal_to_input(src)


def test_relayout_tma_64gib(swz, orc, big):
    """The TMA 128-byte mode on 64 GiB (2^29 rows of the mode's span)."""
    src, dst = big
    _fill(src)
    n = N_BYTES // 2
    assert swz.swz_relayout_tma_path(dst, src, n // 4096, 64, 64, 2, 3, 3, 3, 0) == 3
    _check_relayout(swz, orc, swz.swz_relayout_tma, src, dst, n // 4096, 4096, 2, 3, 3, 3, seed=7)


def test_relayout_staged_and_unaligned_large(swz, orc, big):
    """Ragged 24-byte tiles through the staged kernel, and 16-bit tiles on
    pointers off 16-byte alignment, over 32 GiB (block and chunk indices past
    2^32 bytes)."""
    src, dst = big
    _fill(src)
    half = N_BYTES // 2
    # 24-byte tiles of bytes under Swizzle<1,2,3> (periods of 64 elements do not fit: tile-local, staged)
    n_tiles = half // 24
    _check_relayout(swz, orc, swz.swz_relayout, src[:n_tiles * 24], dst[:n_tiles * 24], n_tiles, 24, 1, 1, 2, 3,
                    seed=8)
    # 64 x 64 16-bit tiles, source 2 bytes and destination 6 bytes off 16-byte alignment
    n_tiles = half // 8192 - 1
    nb = n_tiles * 8192
    _check_relayout(swz, orc, swz.swz_relayout, src[2:2 + nb], dst[6:6 + nb], n_tiles, 4096, 2, 3, 3, 3, seed=9)


def test_bank_profile_and_slice_collision_large(swz, orc, big):
    """The bank profiler over 2^27 patterns (16 GiB of addresses, pattern
    words past 2^32) and the batched slice collision over 2^32 masks (32 GiB
    in, 32 GiB out), each checked at sampled entries, the last included."""
    src, dst = big
    _fill(src)
    # patterns: 32 byte addresses each, made 4-byte aligned below 228 KiB
    n_pat = 1 << 27
    addrs = src[:n_pat * 128].view(torch.int32)
    addrs.bitwise_and_(0x3FFFC)
    addrs.remainder_(228 * 1024)
    ways = dst[:n_pat * 4].view(torch.int32)
    wf = dst[n_pat * 4:n_pat * 8].view(torch.int32)
    swz.swz_bank_profile(addrs, None, n_pat, 4, ways, wf)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    rows = np.sort(rng.choice(n_pat, 4096, replace=False)).astype(np.int64)
    rows[-1] = n_pat - 1
    tr = torch.from_numpy(rows).cuda()
    host = addrs.view(-1, 32)[tr].cpu().numpy().view(np.uint32)
    w_want, f_want = orc.bank_profile(host, 4)
    assert np.array_equal(ways[tr].cpu().numpy(), w_want)
    assert np.array_equal(wf[tr].cpu().numpy(), f_want)
    # slice collision: C = A & ~sw(A) on 2^32 masks, Swizzle<3,4,3>
    n_m = 1 << 32
    A = src[:n_m * 8].view(torch.int64)
    C = dst[:n_m * 8].view(torch.int64)
    swz.swz_slice_collision_batch(A, n_m, 3, 4, 3, C)
    torch.cuda.synchronize()
    idx = np.sort(rng.choice(n_m, 4096, replace=False)).astype(np.int64)
    idx[-1] = n_m - 1
    ti = torch.from_numpy(idx).cuda()
    a = A[ti].cpu().numpy().view(np.uint64)
    want = np.array([orc.slice_collision(int(x), B=3, M=4, S=3) for x in a], dtype=np.uint64)
    assert np.array_equal(C[ti].cpu().numpy().view(np.uint64), want)


def test_transpose_relayout_32gib(swz, orc, big):
    """The transpose fused with the Swizzle<3,4,3> relayout into 128 x 64 tiles,
    on a 131072 x 131072 bf16 matrix (32 GiB): element (r, c) lands at the
    forward relayout position of its transposed offset c * R + r; 2^16 sampled
    elements checked, the last one included."""
    src, dst = big
    R = C = 131072
    te = 128 * 64
    s16 = src[:R * C * 2].view(torch.int16)
    d16 = dst[:R * C * 2].view(torch.int16)
    swz.swz_transpose_relayout(d16, s16, R, C, 2, te, 3, 4, 3)
    torch.cuda.synchronize()
    rng = np.random.default_rng(12)
    r = rng.integers(0, R, 1 << 16).astype(np.int64)
    c = rng.integers(0, C, 1 << 16).astype(np.int64)
    r[-1], c[-1] = R - 1, C - 1
    pos = orc.relayout_positions(c * R + r, tile_elems=te, B=3, M=4, S=3)
    assert torch.equal(d16[torch.from_numpy(pos).cuda()], s16[torch.from_numpy(r * C + c).cuda()])
