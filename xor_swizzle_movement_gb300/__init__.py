"""xor_swizzle_movement_gb300 -- XOR-swizzle data movement on GB300 (sm_103a).

A thin ctypes binding over libswz.so, whose C ABI is declared in
include/swz.h.  Each function here has the name of the C entry point it
calls and only marshals arguments (torch tensors or raw device pointers,
the current torch stream); every step of the work runs in the library's CUDA
kernels.  There is no CPU fallback: if the library has not been built, the
first call raises.

Swizzle<B, M, S>(x) = x ^ (((x >> (M + S)) & ((1 << B) - 1)) << M), with B, M,
S in element-offset units ("CuTe Swizzle 学习手册", section "Swizzle 数学公式").
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "SwzError", "lib", "library_path",
    "swz_relayout", "swz_relayout_tma", "swz_relayout_tma_path", "swz_transpose", "swz_transpose_relayout", "swz_bank_profile", "swz_slice_collision",
    "swz_slice_collision_batch", "swz_slice_layout", "swz_layout_text", "swz_apply", "swz_device_status", "swz_selftest_tma_timeout",
    "swz_transpose_tma_noalloc", "swz_selftest_noalloc_timeout", "swz_staging_probe",
    "swz_status_string", "swz_version",
    "SWZ_OK", "SWZ_ERR_NULL", "SWZ_ERR_PARAM", "SWZ_ERR_SHAPE", "SWZ_ERR_ALIGN", "SWZ_ERR_ALIAS",
    "SWZ_ERR_CUDA", "SWZ_ERR_TIMEOUT", "SWZ_ERR_UNSUPPORTED",
    "SWZ_T_SWIZZLED", "SWZ_T_UNSWIZZLED", "SWZ_T_PADDED", "SWZ_T_TMA",
]

SWZ_OK = 0
SWZ_ERR_NULL = 1
SWZ_ERR_PARAM = 2
SWZ_ERR_SHAPE = 3
SWZ_ERR_ALIGN = 4
SWZ_ERR_ALIAS = 5
SWZ_ERR_CUDA = 6
SWZ_ERR_TIMEOUT = 7
SWZ_ERR_UNSUPPORTED = 8

SWZ_T_SWIZZLED = 0
SWZ_T_UNSWIZZLED = 1
SWZ_T_PADDED = 2
SWZ_T_TMA = 3

_PKG = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_PKG, "_build", "libswz.so")


class SwzError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {swz_status_string(status)} ({status})")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libswz.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libswz.so is not built ({path}); run __graft_entry__.build() "
                               "or python -m xor_swizzle_movement_gb300.build")
        L = ctypes.CDLL(path)
        i32, i64, u64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
        L.swz_relayout.argtypes = [vp, vp, i64, i64, i64, i32, i32, i32, i32, i32, vp]
        L.swz_relayout.restype = i32
        L.swz_relayout_tma.argtypes = [vp, vp, i64, i64, i64, i32, i32, i32, i32, i32, vp]
        L.swz_relayout_tma.restype = i32
        L.swz_transpose.argtypes = [vp, vp, i64, i64, i32, i32, vp]
        L.swz_transpose.restype = i32
        L.swz_transpose_relayout.argtypes = [vp, vp, i64, i64, i32, i64, i32, i32, i32, vp]
        L.swz_transpose_relayout.restype = i32
        L.swz_bank_profile.argtypes = [vp, vp, i64, i32, vp, vp, vp]
        L.swz_bank_profile.restype = i32
        L.swz_slice_collision.argtypes = [u64, i32, i32, i32, ctypes.POINTER(u64)]
        L.swz_slice_collision.restype = i32
        L.swz_slice_layout.argtypes = [u64, i32, i32, i32, ctypes.POINTER(u64), ctypes.POINTER(i32)]
        L.swz_slice_layout.restype = i32
        L.swz_slice_collision_batch.argtypes = [vp, i64, i32, i32, i32, vp, vp]
        L.swz_slice_collision_batch.restype = i32
        L.swz_layout_text.argtypes = [ctypes.c_char_p, i64, i64, i64, i32, i32, i32, i32]
        L.swz_layout_text.restype = i64
        L.swz_apply.argtypes = [u64, i32, i32, i32]
        L.swz_apply.restype = u64
        L.swz_device_status.argtypes = [vp]
        L.swz_device_status.restype = i32
        L.swz_selftest_tma_timeout.argtypes = [vp, vp, i64, i64, u64, vp]
        L.swz_selftest_tma_timeout.restype = i32
        L.swz_relayout_tma_path.argtypes = [vp, vp, i64, i64, i64, i32, i32, i32, i32, i32]
        L.swz_relayout_tma_path.restype = i32
        L.swz_transpose_tma_noalloc.argtypes = [vp, vp, i64, i64, ctypes.POINTER(ctypes.c_uint32), vp]
        L.swz_transpose_tma_noalloc.restype = i32
        L.swz_selftest_noalloc_timeout.argtypes = [vp, vp, i64, i64, u64, ctypes.POINTER(ctypes.c_uint32), vp]
        L.swz_selftest_noalloc_timeout.restype = i32
        L.swz_staging_probe.argtypes = [i32, i32, i32, vp, vp, i64, vp, i64, vp]
        L.swz_staging_probe.restype = i32
        L.swz_status_string.argtypes = [i32]
        L.swz_status_string.restype = ctypes.c_char_p
        L.swz_version.argtypes = []
        L.swz_version.restype = i32
        _lib = L
    return _lib


def _ptr(x) -> int | None:
    """A device pointer from a CUDA tensor (must be contiguous), an int or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != SWZ_OK:
        raise SwzError(status, what)


def swz_relayout(dst, src, n_tiles: int, rows: int, cols: int, esize: int, B: int, M: int, S: int,
                 direction: int, stream=None) -> None:
    """direction 0: dst[t][sw(i)] = src[t][i]; 1: dst[t][i] = src[t][sw(i)]."""
    _check(lib().swz_relayout(_ptr(dst), _ptr(src), n_tiles, rows, cols, esize, B, M, S, direction,
                              _stream(stream)), "swz_relayout")


def swz_relayout_tma(dst, src, n_tiles: int, rows: int, cols: int, esize: int, B: int, M: int, S: int,
                     direction: int, stream=None) -> None:
    """swz_relayout through the TMA hardware swizzle where it applies
    (S = 3, M + log2 esize = 4, 1 <= B <= 3); otherwise the same as swz_relayout."""
    _check(lib().swz_relayout_tma(_ptr(dst), _ptr(src), n_tiles, rows, cols, esize, B, M, S, direction,
                                  _stream(stream)), "swz_relayout_tma")


def swz_relayout_tma_path(dst, src, n_tiles: int, rows: int, cols: int, esize: int, B: int, M: int, S: int,
                          direction: int) -> int:
    """0: swz_relayout_tma would run the register kernels; 1..4: the TMA mode
    (32-, 64-, 128-byte, 128-byte with 32-byte atoms); -status for bad arguments."""
    return int(lib().swz_relayout_tma_path(_ptr(dst), _ptr(src), n_tiles, rows, cols, esize, B, M, S, direction))


def swz_transpose(dst, src, rows: int, cols: int, esize: int, variant: int = SWZ_T_SWIZZLED,
                  stream=None) -> None:
    """dst (cols x rows) = transpose of src (rows x cols), raw esize-byte elements."""
    _check(lib().swz_transpose(_ptr(dst), _ptr(src), rows, cols, esize, variant, _stream(stream)),
           "swz_transpose")


def swz_transpose_relayout(dst, src, rows: int, cols: int, esize: int, tile_elems: int, B: int, M: int,
                           S: int, stream=None) -> None:
    """dst = the transpose of src (rows x cols), cut into tiles of tile_elems
    elements, each tile in Swizzle<B,M,S> order (forward relayout)."""
    _check(lib().swz_transpose_relayout(_ptr(dst), _ptr(src), rows, cols, esize, tile_elems, B, M, S,
                                        _stream(stream)), "swz_transpose_relayout")


def swz_bank_profile(byte_addrs, active, n: int, access_bytes: int, ways, wavefronts,
                     stream=None) -> None:
    _check(lib().swz_bank_profile(_ptr(byte_addrs), _ptr(active), n, access_bytes, _ptr(ways),
                                  _ptr(wavefronts), _stream(stream)), "swz_bank_profile")


def swz_slice_collision(A: int, B: int, M: int, S: int) -> int:
    out = ctypes.c_uint64(0)
    _check(lib().swz_slice_collision(A, B, M, S, ctypes.byref(out)), "swz_slice_collision")
    return int(out.value)


def swz_slice_layout(A: int, B: int, M: int, S: int):
    """Per-bit strides of the plain layout equal to the swizzle on slice A, or
    None when the slice collides (A & ~sw(A) != 0)."""
    strides = (ctypes.c_uint64 * 64)()
    n = ctypes.c_int(0)
    status = lib().swz_slice_layout(A, B, M, S, strides, ctypes.byref(n))
    if status == SWZ_ERR_UNSUPPORTED:
        return None
    _check(status, "swz_slice_layout")
    return [int(strides[i]) for i in range(n.value)]


def swz_slice_collision_batch(A, n: int, B: int, M: int, S: int, C, stream=None) -> None:
    _check(lib().swz_slice_collision_batch(_ptr(A), n, B, M, S, _ptr(C), _stream(stream)),
           "swz_slice_collision_batch")


def swz_layout_text(rows: int, cols: int, esize: int, B: int, M: int, S: int) -> str:
    """Text map of a swizzled rows x cols tile: "physical_offset/bank" per element."""
    n = lib().swz_layout_text(None, 0, rows, cols, esize, B, M, S)
    if n < 0:
        raise SwzError(SWZ_ERR_PARAM, "swz_layout_text")
    buf = ctypes.create_string_buffer(int(n) + 1)
    lib().swz_layout_text(buf, n + 1, rows, cols, esize, B, M, S)
    return buf.value.decode()


def swz_apply(x: int, B: int, M: int, S: int) -> int:
    return int(lib().swz_apply(x, B, M, S))


def swz_device_status(stream=None) -> int:
    """Synchronises the stream; returns SWZ_OK or SWZ_ERR_TIMEOUT (does not raise)."""
    return int(lib().swz_device_status(_stream(stream)))


def swz_selftest_tma_timeout(dst, src, rows: int, cols: int, wait_ns: int, stream=None) -> None:
    _check(lib().swz_selftest_tma_timeout(_ptr(dst), _ptr(src), rows, cols, wait_ns, _stream(stream)),
           "swz_selftest_tma_timeout")


def swz_transpose_tma_noalloc(dst, src, rows: int, cols: int, wait: bool = False, stream=None) -> int:
    """The 16-bit TMA transpose with no allocation by the library (for callers
    whose device memory is owned by their own pool).  With wait=True the call
    waits for the stream and returns 1 if a bounded wait gave up, else 0."""
    flag = ctypes.c_uint32(0)
    status = lib().swz_transpose_tma_noalloc(_ptr(dst), _ptr(src), rows, cols,
                                             ctypes.byref(flag) if wait else None, _stream(stream))
    if status == SWZ_ERR_TIMEOUT:
        return 1
    _check(status, "swz_transpose_tma_noalloc")
    return int(flag.value)


def swz_selftest_noalloc_timeout(dst, src, rows: int, cols: int, wait_ns: int, stream=None) -> int:
    """Runs swz_transpose_tma_noalloc's kernel with no copy issued; returns the
    timed_out flag (1 when the expiry was reported) and the status code."""
    flag = ctypes.c_uint32(0)
    status = lib().swz_selftest_noalloc_timeout(_ptr(dst), _ptr(src), rows, cols, wait_ns, ctypes.byref(flag),
                                                _stream(stream))
    if status != SWZ_ERR_TIMEOUT:
        _check(status, "swz_selftest_noalloc_timeout")
    return int(flag.value), int(status)


def swz_staging_probe(esize: int, variant: int, iters: int, ctas: int, gsrc=None, gdst=None, gbytes: int = 0,
                      sink=None, stream=None) -> None:
    """Fill and drain one transpose staging `iters` times per CTA on register
    data (a diagnostic for the shared-memory bank-conflict counters); with
    gsrc / gdst, 16-byte global traffic streams alongside."""
    _check(lib().swz_staging_probe(esize, variant, iters, _ptr(gsrc), _ptr(gdst), gbytes, _ptr(sink), ctas,
                                   _stream(stream)), "swz_staging_probe")


def swz_status_string(status: int) -> str:
    try:
        return lib().swz_status_string(status).decode()
    except Exception:  # the library itself is missing
        return f"status {status}"


def swz_version() -> int:
    return int(lib().swz_version())
