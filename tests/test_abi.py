"""The C ABI without a GPU: the library loads, exports every function that
include/swz.h declares, its host functions agree with the oracle, and every
invalid request is rejected with its status code before anything is
launched (the pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def swz():
    import xor_swizzle_movement_gb300 as m
    if not os.path.exists(m.library_path()):
        from xor_swizzle_movement_gb300 import build
        build.build()
    m.lib()
    return m


def declared_functions():
    text = open(os.path.join(ROOT, "include", "swz.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swz_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_function(swz):
    names = declared_functions()
    assert {"swz_relayout", "swz_transpose", "swz_bank_profile", "swz_slice_collision"} <= set(names)
    for name in names:
        assert hasattr(swz.lib(), name), name
        assert hasattr(swz, name), name  # the binding has the same names


def test_apply_matches_oracle(swz, orc):
    for (B, M, S) in [(5, 0, 6), (3, 3, 3), (3, 4, 3), (2, 0, 1), (4, 4, 11), (0, 3, 3),
                      (3, 4, -10), (2, 0, -1), (3, 1, -2), (5, 2, -5), (4, 0, -7)]:
        for x in list(range(0, 5000, 7)) + [673, 2**40 + 12345]:
            assert swz.swz_apply(x, B, M, S) == orc.swizzle(x, B=B, M=M, S=S)


def test_slice_collision_host(swz, orc):
    for (B, M, S) in [(3, 2, 4), (2, 0, 1), (3, 1, 2), (5, 0, 5), (3, 2, -4), (2, 0, -1), (3, 1, -2)]:
        for A in range(1 << (B + M + S + 1)):
            assert swz.swz_slice_collision(A, B, M, S) == orc.slice_collision(A, B=B, M=M, S=S)
    with pytest.raises(swz.SwzError) as e:
        swz.swz_slice_collision(1, 3, 0, 0, )
    assert e.value.status == swz.SWZ_ERR_PARAM
    assert swz.lib().swz_slice_collision(1, 3, 0, 3, None) == swz.SWZ_ERR_NULL


FAKE_A, FAKE_B = 1 << 40, 1 << 41  # never dereferenced: every case below fails validation


@pytest.mark.parametrize("args,status", [
    ((FAKE_B, FAKE_A, 1, 8, 8, 3, 3, 0, 3, 0), "SWZ_ERR_PARAM"),      # esize 3
    ((FAKE_B, FAKE_A, 1, 8, 8, 2, 3, 0, 0, 0), "SWZ_ERR_PARAM"),      # S = 0
    ((FAKE_B, FAKE_A, 1, 8, 8, 2, 17, 0, 1, 0), "SWZ_ERR_PARAM"),     # B > 16
    ((FAKE_B, FAKE_A, 1, 8, 8, 2, 3, 0, 3, 2), "SWZ_ERR_PARAM"),      # direction
    ((FAKE_B, FAKE_A, 1, 8, 8, 2, 16, 16, 17, 0), "SWZ_ERR_PARAM"),   # B + M + S > 48
    ((FAKE_B, FAKE_A, 1, 8, 8, 2, 3, 0, -33, 0), "SWZ_ERR_PARAM"),    # |S| > 32
    ((FAKE_B, FAKE_A, 1, 8, 8, 2, 16, 16, -17, 0), "SWZ_ERR_PARAM"),  # B + M + |S| > 48
    ((FAKE_B, FAKE_A, 1, 8, 8, 2, 3, 0, -4, 0), "SWZ_ERR_SHAPE"),     # 64 % 2^(0 + 4 + 3) != 0
    ((FAKE_B, FAKE_A, -1, 8, 8, 2, 3, 0, 3, 0), "SWZ_ERR_SHAPE"),
    ((FAKE_B, FAKE_A, 1, 3, 4, 2, 2, 2, 2, 0), "SWZ_ERR_SHAPE"),      # tile not closed
    ((FAKE_B, FAKE_A, 2**40, 2**20, 2**20, 2, 3, 0, 3, 0), "SWZ_ERR_SHAPE"),  # overflow
    ((0, FAKE_A, 1, 8, 8, 2, 3, 0, 3, 0), "SWZ_ERR_NULL"),
    ((FAKE_B + 1, FAKE_A, 1, 8, 8, 2, 3, 0, 3, 0), "SWZ_ERR_ALIGN"),
    ((FAKE_A + 64, FAKE_A, 1, 8, 8, 2, 3, 0, 3, 0), "SWZ_ERR_ALIAS"),
])
def test_relayout_validation(swz, args, status):
    assert swz.lib().swz_relayout(*args, None) == getattr(swz, status)


@pytest.mark.parametrize("args,status", [
    ((FAKE_B, FAKE_A, 8, 8, 3, 0), "SWZ_ERR_PARAM"),
    ((FAKE_B, FAKE_A, 8, 8, 4, 4), "SWZ_ERR_PARAM"),
    ((FAKE_B, FAKE_A, 8, 8, 4, 3), "SWZ_ERR_PARAM"),
    ((FAKE_B, FAKE_A, -8, 8, 4, 0), "SWZ_ERR_SHAPE"),
    ((FAKE_B, 0, 8, 8, 4, 0), "SWZ_ERR_NULL"),
    ((FAKE_B + 2, FAKE_A, 8, 8, 4, 0), "SWZ_ERR_ALIGN"),
    ((FAKE_A, FAKE_A, 8, 8, 4, 0), "SWZ_ERR_ALIAS"),
])
def test_transpose_validation(swz, args, status):
    assert swz.lib().swz_transpose(*args, None) == getattr(swz, status)


def test_empty_requests_succeed(swz):
    L = swz.lib()
    assert L.swz_relayout(0, 0, 0, 8, 8, 2, 3, 0, 3, 0, None) == swz.SWZ_OK
    assert L.swz_transpose(0, 0, 0, 8, 4, 0, None) == swz.SWZ_OK
    assert L.swz_bank_profile(0, 0, 0, 4, 0, 0, None) == swz.SWZ_OK
    assert L.swz_slice_collision_batch(0, 0, 3, 0, 3, 0, None) == swz.SWZ_OK


def test_bank_profile_validation(swz):
    L = swz.lib()
    assert L.swz_bank_profile(FAKE_A, 0, 4, 3, FAKE_B, FAKE_B + 64, None) == swz.SWZ_ERR_PARAM
    assert L.swz_bank_profile(FAKE_A, 0, -1, 4, FAKE_B, FAKE_B + 64, None) == swz.SWZ_ERR_SHAPE
    assert L.swz_bank_profile(FAKE_A, 0, 4, 4, 0, FAKE_B, None) == swz.SWZ_ERR_NULL
    assert L.swz_bank_profile(FAKE_A + 1, 0, 4, 4, FAKE_B, FAKE_B + 64, None) == swz.SWZ_ERR_ALIGN


def test_status_strings(swz):
    for code in range(9):
        s = swz.swz_status_string(code)
        assert s.startswith("SWZ_")
    assert "unknown" in swz.swz_status_string(99)
    assert swz.swz_version() >= 100


@pytest.mark.parametrize("B,M,S", [(2, 0, 2), (3, 1, 2), (2, 1, 3), (3, 0, 1), (2, 0, -2), (3, 1, -2), (3, 0, -1)])
def test_slice_layout(swz, orc, B, M, S):
    """Slices whose collision mask is 0 come back as per-bit strides that
    reproduce the swizzle on every subset (the oracle's brute force agrees);
    the others are refused."""
    import itertools
    for A in range(1 << (B + M + abs(S) + 1)):
        strides = swz.swz_slice_layout(A, B, M, S)
        assert (strides is not None) == orc.slice_is_layout(A, B=B, M=M, S=S), A
        if strides is None:
            continue
        bits = [i for i in range(64) if (A >> i) & 1]
        assert len(strides) == len(bits)
        for pick in itertools.product((0, 1), repeat=len(bits)):
            x = sum(b << i for b, i in zip(pick, bits))
            assert sum(b * st for b, st in zip(pick, strides)) == orc.swizzle(x, B=B, M=M, S=S)


def test_layout_text_matches_oracle_dump(swz, orc):
    for (rows, cols, esize, B, M, S) in [(32, 64, 4, 5, 0, 6), (8, 64, 2, 3, 3, 3), (16, 16, 8, 4, 0, 4)]:
        assert swz.swz_layout_text(rows, cols, esize, B, M, S) == orc.dump_layout(rows, cols, esize, B=B, M=M, S=S)
    assert swz.lib().swz_layout_text(None, 0, -1, 4, 4, 3, 0, 3) == -1
    # truncation: the returned length is the whole text, the buffer holds a prefix
    import ctypes
    full = swz.swz_layout_text(4, 4, 4, 2, 0, 2)
    buf = ctypes.create_string_buffer(10)
    assert swz.lib().swz_layout_text(buf, 10, 4, 4, 4, 2, 0, 2) == len(full)
    assert buf.value.decode() == full[:9]


def test_relayout_tma_path_reports_argument_errors(swz):
    """The path query validates like swz_relayout_tma and returns -status."""
    a, b = 1 << 20, 1 << 21   # never dereferenced
    assert swz.swz_relayout_tma_path(a, b, 4, 64, 64, 2, 3, 3, 0, 0) == -swz.SWZ_ERR_PARAM     # S = 0
    assert swz.swz_relayout_tma_path(a, b, 4, 1, 60, 2, 3, 3, 3, 0) == -swz.SWZ_ERR_SHAPE     # tile not closed
    assert swz.swz_relayout_tma_path(a, a, 4, 64, 64, 2, 3, 3, 3, 0) == -swz.SWZ_ERR_ALIAS
    assert swz.swz_relayout_tma_path(a, b, 0, 64, 64, 2, 3, 3, 3, 0) == 0                     # empty
    assert swz.swz_relayout_tma_path(a + 2, b, 4, 64, 64, 2, 3, 3, 3, 0) == 0                 # misaligned
