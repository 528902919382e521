"""Device-buffer helpers for the GPU parity tests: every output buffer is
surrounded by canary bytes that are checked after the kernel ran."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

GUARD = 512
CANARY = 0xA5


def to_device(arr: np.ndarray, offset: int = 0):
    """Copy arr's bytes to the GPU at byte `offset` past a 512-byte-aligned start.
    Returns (backing, view) as uint8 tensors."""
    b = np.ascontiguousarray(arr).view(np.uint8).ravel()
    full = torch.full((GUARD + offset + b.size + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    view = full[GUARD + offset: GUARD + offset + b.size]
    if b.size:
        view.copy_(torch.from_numpy(b.copy()).to("cuda"))
    return full, view


def empty_device(nbytes: int, offset: int = 0):
    full = torch.full((GUARD + offset + nbytes + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    return full, full[GUARD + offset: GUARD + offset + nbytes]


def to_host(view, dtype, shape=None) -> np.ndarray:
    a = view.cpu().numpy().view(dtype)
    return a.reshape(shape) if shape is not None else a


def guards_intact(full, offset: int, nbytes: int) -> bool:
    h = full.cpu().numpy()
    head = h[:GUARD + offset]
    tail = h[GUARD + offset + nbytes:]
    return bool((head == CANARY).all() and (tail == CANARY).all())


def void_dtype(esize: int):
    return np.dtype(f"V{esize}")
