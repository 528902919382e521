"""CPU oracle for the XOR-swizzle data-movement path -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and it imports nothing
from the product package: the two share no code.

The arithmetic lives in ``swz_oracle.c`` (plain C, one element per loop
iteration); this module only compiles it with gcc and marshals numpy arrays
through ctypes.  The parity status of every function is stated in the C
file's header: every function is pinned (the grouping of 8-byte bank-model
passes into consecutive half-warps is a reading the pins constrain).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swz_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

ORC_OK = 0
ORC_BAD_ARG = 1
ORC_NOT_CLOSED = 2


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, no CUDA)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra",
                           "-o", tmp, _SRC])
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    u64, i64, i32, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    L.orc_swizzle.argtypes = [u64, i32, i32, i32]
    L.orc_swizzle.restype = u64
    L.orc_relayout.argtypes = [vp, vp, i64, i64, i32, i32, i32, i32, i32]
    L.orc_relayout.restype = i32
    L.orc_relayout_positions.argtypes = [vp, i64, i64, i32, i32, i32, vp]
    L.orc_relayout_positions.restype = i32
    L.orc_transpose.argtypes = [vp, vp, i64, i64, i32]
    L.orc_transpose.restype = i32
    L.orc_transpose_relayout.argtypes = [vp, vp, vp, i64, i64, i32, i64, i32, i32, i32]
    L.orc_transpose_relayout.restype = i32
    L.orc_bank_profile.argtypes = [vp, vp, i64, i32, vp, vp]
    L.orc_bank_profile.restype = i32
    L.orc_slice_collision.argtypes = [u64, i32, i32, i32]
    L.orc_slice_collision.restype = u64
    L.orc_slice_is_layout.argtypes = [u64, i32, i32, i32]
    L.orc_slice_is_layout.restype = i32
    L.orc_dump_layout.argtypes = [ctypes.c_char_p, i64, i64, i64, i32, i32, i32, i32]
    L.orc_dump_layout.restype = i64
    return L


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


class Oracle:
    """The oracle's functions bound to one compiled copy of it.  The
    module-level functions use the default build; the tests that plant
    mistakes in a copy of the C source bind that copy here."""

    def __init__(self, path: str):
        self.L = _bind(path)

    def swizzle(self, offset, **kw):
        return _swizzle(self.L, offset, **kw)

    def relayout(self, src, **kw):
        return _relayout(self.L, src, **kw)

    def relayout_positions(self, idx, **kw):
        return _relayout_positions(self.L, idx, **kw)

    def transpose(self, src):
        return _transpose(self.L, src)

    def transpose_relayout(self, src, **kw):
        return _transpose_relayout(self.L, src, **kw)

    def bank_profile(self, addrs, width, active=None):
        return _bank_profile(self.L, addrs, width, active)

    def slice_collision(self, A, **kw):
        return _slice_collision(self.L, A, **kw)

    def slice_is_layout(self, A, **kw):
        return _slice_is_layout(self.L, A, **kw)

    def dump_layout(self, rows, cols, esize, **kw):
        return _dump_layout(self.L, rows, cols, esize, **kw)


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# The oracle follows the pages' own argument order: swizzle<base, bits, shift>,
# i.e. (M, B, S).  The wrappers below take keyword arguments B, M, S so that a
# caller cannot mix the orders up.

def _swizzle(L, offset: int, *, B: int, M: int, S: int) -> int:
    return int(L.orc_swizzle(offset, M, B, S))


def _relayout(L, src: np.ndarray, *, tile_elems: int, B: int, M: int, S: int,
              direction: int) -> np.ndarray:
    """src: contiguous array whose size is a multiple of tile_elems elements."""
    src = np.ascontiguousarray(src)
    dst = np.empty_like(src)
    esize = src.dtype.itemsize
    n_tiles = src.size // tile_elems if tile_elems else 0
    assert n_tiles * tile_elems == src.size
    rc = L.orc_relayout(_ptr(dst), _ptr(src), n_tiles, tile_elems, esize, M, B, S, direction)
    if rc != ORC_OK:
        raise ValueError(f"orc_relayout failed with {rc}")
    return dst


def _relayout_positions(L, idx: np.ndarray, *, tile_elems: int, B: int, M: int, S: int) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty_like(idx)
    rc = L.orc_relayout_positions(_ptr(idx), idx.size, tile_elems, M, B, S, _ptr(out))
    if rc != ORC_OK:
        raise ValueError(f"orc_relayout_positions failed with {rc}")
    return out


def _transpose(L, src: np.ndarray) -> np.ndarray:
    """src: 2-D contiguous array; returns its transpose as a new contiguous array."""
    src = np.ascontiguousarray(src)
    rows, cols = src.shape
    dst = np.empty((cols, rows), dtype=src.dtype)
    rc = L.orc_transpose(_ptr(dst), _ptr(src), rows, cols, src.dtype.itemsize)
    if rc != ORC_OK:
        raise ValueError(f"orc_transpose failed with {rc}")
    return dst


def _transpose_relayout(L, src: np.ndarray, *, tile_elems: int, B: int, M: int, S: int) -> np.ndarray:
    """src: 2-D contiguous (rows, cols); returns the flat cols*rows result."""
    src = np.ascontiguousarray(src)
    rows, cols = src.shape
    dst = np.empty(rows * cols, dtype=src.dtype)
    tmp = np.empty(rows * cols, dtype=src.dtype)
    rc = L.orc_transpose_relayout(_ptr(dst), _ptr(src), _ptr(tmp), rows, cols, src.dtype.itemsize,
                                  tile_elems, M, B, S)
    if rc != ORC_OK:
        raise ValueError(f"orc_transpose_relayout failed with {rc}")
    return dst


def _bank_profile(L, addrs: np.ndarray, width: int, active: np.ndarray | None = None):
    """addrs: (n, 32) uint32 byte addresses. Returns (ways, wavefronts) int32 arrays."""
    addrs = np.ascontiguousarray(addrs, dtype=np.uint32).reshape(-1, 32)
    n = addrs.shape[0]
    ways = np.empty(n, dtype=np.int32)
    wf = np.empty(n, dtype=np.int32)
    act_ptr = None
    if active is not None:
        active = np.ascontiguousarray(active, dtype=np.uint32)
        assert active.shape == (n,)
        act_ptr = _ptr(active)
    rc = L.orc_bank_profile(_ptr(addrs), act_ptr, n, width, _ptr(ways), _ptr(wf))
    if rc != ORC_OK:
        raise ValueError(f"orc_bank_profile failed with {rc}")
    return ways, wf


def _slice_collision(L, A: int, *, B: int, M: int, S: int) -> int:
    return int(L.orc_slice_collision(A, M, B, S))


def _slice_is_layout(L, A: int, *, B: int, M: int, S: int) -> bool:
    return bool(L.orc_slice_is_layout(A, M, B, S))


def _dump_layout(L, rows: int, cols: int, esize: int, *, B: int, M: int, S: int) -> str:
    n = L.orc_dump_layout(None, 0, rows, cols, esize, M, B, S)
    buf = ctypes.create_string_buffer(int(n) + 1)
    L.orc_dump_layout(buf, n + 1, rows, cols, esize, M, B, S)
    return buf.value.decode()


# module-level functions on the default build
def swizzle(offset, **kw):
    return _swizzle(lib(), offset, **kw)


def relayout(src, **kw):
    return _relayout(lib(), src, **kw)


def relayout_positions(idx, **kw):
    return _relayout_positions(lib(), idx, **kw)


def transpose(src):
    return _transpose(lib(), src)


def transpose_relayout(src, **kw):
    return _transpose_relayout(lib(), src, **kw)


def bank_profile(addrs, width, active=None):
    return _bank_profile(lib(), addrs, width, active)


def slice_collision(A, **kw):
    return _slice_collision(lib(), A, **kw)


def slice_is_layout(A, **kw):
    return _slice_is_layout(lib(), A, **kw)


def dump_layout(rows, cols, esize, **kw):
    return _dump_layout(lib(), rows, cols, esize, **kw)


def compile_copy(c_source: str, out_dir: str) -> str:
    """Compile a (possibly edited) copy of the oracle's C source; returns the
    shared library's path.  Used by the tests that plant mistakes."""
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, "swz_oracle_copy.c")
    with open(src, "w") as f:
        f.write(c_source)
    out = os.path.join(out_dir, "liboracle_copy.so")
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-o", out, src])
    return out


def c_source() -> str:
    with open(_SRC) as f:
        return f.read()
