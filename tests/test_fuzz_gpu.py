"""Seeded random parity sweep: many small relayout, transpose and fused
requests with random parameters (negative shifts included), shapes and
pointer offsets, each compared bit for bit with the CPU oracle.  Every
request is valid; together they reach every kernel path (vector, misaligned
vector, fixed lane map, staged, element by element, TMA modes, each
transpose staging)."""
import math

import numpy as np
import pytest

from gpu_util import empty_device, guards_intact, to_device, to_host, torch, void_dtype

pytestmark = pytest.mark.gpu

ESIZES = [1, 2, 4, 8, 16]


@pytest.fixture(scope="module")
def swz():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import xor_swizzle_movement_gb300 as m
    m.lib()
    return m


def random_relayout(rng):
    """A valid relayout request: (esize, n_tiles, rows, cols, B, M, S, direction, offsets)."""
    esize = int(rng.choice(ESIZES))
    B = int(rng.integers(0, 5))
    M = int(rng.integers(0, 5))
    S = int(rng.integers(1, 8)) * (-1 if rng.random() < 0.3 else 1)
    # tiles close under the swizzle in blocks of 2^(bit above the written field)
    unit = 1 << (M + B + (-S if S < 0 else 0))
    # tile: a multiple of 2^(M+B) elements, up to ~4096
    mult = int(rng.integers(1, max(2, 4096 // unit) + 1))
    tile = unit * mult
    # split the tile into rows x cols
    divs = [d for d in range(1, min(tile, 256) + 1) if tile % d == 0]
    rows = int(rng.choice(divs))
    cols = tile // rows
    n_tiles = int(rng.integers(1, max(2, (1 << 18) // (tile * esize)) + 1))
    direction = int(rng.integers(0, 2))
    aligned = rng.random() < 0.7
    src_off = 0 if aligned else esize * int(rng.integers(1, 16 // esize + 1)) % 16
    dst_off = 0 if aligned else esize * int(rng.integers(0, 16 // esize + 1)) % 16
    return esize, n_tiles, rows, cols, B, M, S, direction, src_off, dst_off


@pytest.mark.parametrize("block", range(6))
def test_relayout_fuzz(swz, orc, block):
    from xor_swizzle_movement_gb300 import inputs
    rng = np.random.default_rng(1000 + block)
    for case in range(40):
        esize, n_tiles, rows, cols, B, M, S, direction, so, do = random_relayout(rng)
        tile = rows * cols
        host = inputs.random_bytes(n_tiles * tile * esize, seed=block * 100 + case).view(void_dtype(esize))
        _, src = to_device(host, so)
        full, dst = empty_device(host.nbytes, do)
        tma = rng.random() < 0.3
        fn = swz.swz_relayout_tma if tma else swz.swz_relayout
        fn(dst, src, n_tiles, rows, cols, esize, B, M, S, direction)
        torch.cuda.synchronize()
        assert guards_intact(full, do, host.nbytes)
        got = to_host(dst, host.dtype)
        want = orc.relayout(host, tile_elems=tile, B=B, M=M, S=S, direction=direction)
        assert got.tobytes() == want.tobytes(), (esize, n_tiles, rows, cols, B, M, S, direction, so, do, tma)


@pytest.mark.parametrize("block", range(4))
def test_relayout_fuzz_16_byte_offsets(swz, orc, block):
    """Requests on pointers 16-byte aligned but, at random, not 32-byte aligned
    (offsets 0, 16, 32 or 48 bytes from a 512-byte boundary), half of them with
    negative shifts: the kernels that move 32 bytes per access must fall back
    when either pointer is off 32-byte alignment."""
    from xor_swizzle_movement_gb300 import inputs
    rng = np.random.default_rng(5000 + block)
    for case in range(40):
        esize, n_tiles, rows, cols, B, M, S, direction, _, _ = random_relayout(rng)
        if rng.random() < 0.5 and S > 0:
            S = -S
            unit = 1 << (M + B - S)
            tile = rows * cols
            if tile % unit:
                rows, cols = 1, unit * max(1, tile // unit)
        tile = rows * cols
        so, do = (int(x) for x in rng.choice([0, 16, 32, 48], size=2))
        host = inputs.random_bytes(n_tiles * tile * esize, seed=7000 + block * 100 + case).view(void_dtype(esize))
        _, src = to_device(host, so)
        full, dst = empty_device(host.nbytes, do)
        swz.swz_relayout(dst, src, n_tiles, rows, cols, esize, B, M, S, direction)
        torch.cuda.synchronize()
        assert guards_intact(full, do, host.nbytes)
        got = to_host(dst, host.dtype)
        want = orc.relayout(host, tile_elems=tile, B=B, M=M, S=S, direction=direction)
        assert got.tobytes() == want.tobytes(), (esize, n_tiles, rows, cols, B, M, S, direction, so, do)


@pytest.mark.parametrize("block", range(3))
def test_relayout_fuzz_wide_parameters(swz, orc, block):
    """Wider swizzles than the sweep's ranges (B up to 8, M up to 5, |S| up to
    12, mostly negative): closure blocks up to 2^17 elements, where the
    negative shifts reach the register coset kernels' slot and block-store
    forms, lane maps with larger g, and the warp kernel's bigger blocks."""
    from xor_swizzle_movement_gb300 import inputs
    rng = np.random.default_rng(9000 + block)
    for case in range(30):
        esize = int(rng.choice([1, 2, 4, 8]))
        lv = {1: 4, 2: 3, 4: 2, 8: 1}[esize]
        B = int(rng.integers(1, 9))
        M = int(rng.integers(0, lv + 1))              # mostly below log2 V: vectors split
        S = int(rng.integers(1, 4) if rng.random() < 0.5 else rng.integers(1, 13))
        S = -S if rng.random() < 0.75 else S
        hi = (M - S + B) if S < 0 else (M + B)       # tiles close under sw in blocks of 2^hi
        if hi > 17:
            continue
        tile = (1 << hi) * int(rng.integers(1, 4))
        n_tiles = max(1, min(64, (4 << 20) // (tile * esize)))
        direction = int(rng.integers(0, 2))
        so, do = (int(x) for x in rng.choice([0, 16, 32], size=2))
        host = inputs.random_bytes(n_tiles * tile * esize, seed=9500 + block * 100 + case).view(void_dtype(esize))
        _, src = to_device(host, so)
        full, dst = empty_device(host.nbytes, do)
        swz.swz_relayout(dst, src, n_tiles, 1, tile, esize, B, M, S, direction)
        torch.cuda.synchronize()
        assert guards_intact(full, do, host.nbytes)
        got = to_host(dst, host.dtype)
        want = orc.relayout(host, tile_elems=tile, B=B, M=M, S=S, direction=direction)
        assert got.tobytes() == want.tobytes(), (esize, n_tiles, tile, B, M, S, direction, so, do)


def test_relayout_tma_modes_fuzz(swz, orc):
    """Requests inside the TMA's hardware modes (Sw<B, 4 - log2 e, 3>, tiles of
    whole 2^(B+7)-byte periods) with random tile and buffer sizes."""
    from xor_swizzle_movement_gb300 import inputs
    rng = np.random.default_rng(77)
    for case in range(40):
        esize = int(rng.choice([1, 2, 4, 8, 16]))
        B = int(rng.integers(1, 4))
        M = 4 - int(math.log2(esize))
        period = 1 << (B + 7)
        tile_bytes = period * int(rng.integers(1, 9))
        n_tiles = int(rng.integers(1, 40))
        tile = tile_bytes // esize
        cols = max(1, 128 // esize)
        rows = tile // cols if tile % cols == 0 else 1
        cols = tile // rows
        host = inputs.random_bytes(n_tiles * tile_bytes, seed=500 + case).view(void_dtype(esize))
        _, src = to_device(host, 0)
        full, dst = empty_device(host.nbytes, 0)
        direction = int(rng.integers(0, 2))
        swz.swz_relayout_tma(dst, src, n_tiles, rows, cols, esize, B, M, 3, direction)
        torch.cuda.synchronize()
        assert guards_intact(full, 0, host.nbytes)
        got = to_host(dst, host.dtype)
        want = orc.relayout(host, tile_elems=tile, B=B, M=M, S=3, direction=direction)
        assert got.tobytes() == want.tobytes(), (esize, B, tile_bytes, n_tiles, direction)
    assert swz.swz_device_status() == swz.SWZ_OK


@pytest.mark.parametrize("block", range(4))
def test_transpose_fuzz(swz, orc, block):
    from xor_swizzle_movement_gb300 import inputs
    rng = np.random.default_rng(2000 + block)
    for case in range(40):
        esize = int(rng.choice(ESIZES))
        rows = int(rng.integers(1, 600))
        cols = int(rng.integers(1, 600))
        variants = [swz.SWZ_T_SWIZZLED, swz.SWZ_T_UNSWIZZLED, swz.SWZ_T_PADDED] + ([swz.SWZ_T_TMA] if esize == 2 else [])
        variant = int(rng.choice(variants))
        aligned = rng.random() < 0.7
        so = 0 if aligned else esize * int(rng.integers(1, 16 // esize + 1)) % 16
        do = 0 if aligned else esize * int(rng.integers(0, 16 // esize + 1)) % 16
        host = inputs.random_bytes(rows * cols * esize, seed=3000 + block * 100 + case)
        host = host.view(void_dtype(esize)).reshape(rows, cols)
        _, src = to_device(host, so)
        full, dst = empty_device(host.nbytes, do)
        swz.swz_transpose(dst, src, rows, cols, esize, variant)
        torch.cuda.synchronize()
        assert guards_intact(full, do, host.nbytes)
        got = to_host(dst, host.dtype, (cols, rows))
        assert got.tobytes() == orc.transpose(host).tobytes(), (esize, rows, cols, variant, so, do)
    assert swz.swz_device_status() == swz.SWZ_OK


@pytest.mark.parametrize("block", range(3))
def test_transpose_relayout_fuzz(swz, orc, block):
    from xor_swizzle_movement_gb300 import inputs
    rng = np.random.default_rng(4000 + block)
    done = 0
    while done < 30:
        esize = int(rng.choice(ESIZES))
        B, M, S = int(rng.integers(0, 4)), int(rng.integers(0, 4)), int(rng.integers(1, 6))
        if rng.random() < 0.3:
            S = -S
        unit = 1 << (M + B + (-S if S < 0 and B > 0 else 0))
        rows = int(rng.integers(1, 300))
        cols = int(rng.integers(1, 300))
        n = rows * cols
        # a tile size that closes under the swizzle and divides the matrix
        cands = [t for t in range(unit, min(n, 8192) + 1, unit) if n % t == 0]
        if not cands:
            continue
        te = int(rng.choice(cands))
        host = inputs.random_bytes(n * esize, seed=5000 + block * 100 + done).view(void_dtype(esize)).reshape(rows, cols)
        _, src = to_device(host, 0)
        full, dst = empty_device(host.nbytes, 0)
        swz.swz_transpose_relayout(dst, src, rows, cols, esize, te, B, M, S)
        torch.cuda.synchronize()
        assert guards_intact(full, 0, host.nbytes)
        got = to_host(dst, host.dtype)
        want = orc.transpose_relayout(host, tile_elems=te, B=B, M=M, S=S)
        assert got.tobytes() == want.tobytes(), (esize, rows, cols, te, B, M, S)
        done += 1
