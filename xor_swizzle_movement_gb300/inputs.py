"""Seeded synthetic inputs shared by the tests and the benchmark.

This module holds no swizzle, transpose or bank arithmetic: it only draws
random host buffers (torch CPU generator, fixed seeds) with the shapes and
value distributions of the workloads below, so that the CUDA path and the CPU
oracle see the same bytes.

  seed 0  uint16 bit patterns (the 64x64 fp16 tiles of the small relayout case)
  seed 1  N(0,1) values rounded to bf16 (128x64 bf16 tiles)
  seed 2  uniform [-1, 1) fp32 (the fp32 transpose)
  seed 3  uniform fp16 bit patterns with the NaN encodings removed
  seed 4  uniform random bytes (fp64 transpose, int8 tiles, uint16 sweep)
  seed 5  random warp access patterns for the bank profiler
"""
from __future__ import annotations

import numpy as np
import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def random_bytes(nbytes: int, seed: int) -> np.ndarray:
    """Uniform random bytes (uint8)."""
    t = torch.randint(0, 256, (nbytes,), generator=_gen(seed), dtype=torch.uint8)
    return t.numpy()


def uint16_bits(n: int, seed: int = 0) -> np.ndarray:
    """n uniform random 16-bit patterns."""
    return random_bytes(2 * n, seed).view(np.uint16)


def bf16_normal(n: int, seed: int = 1) -> np.ndarray:
    """n values drawn from N(0, 1) in fp32 and rounded to bf16 (round to
    nearest even); returned as their uint16 bit patterns."""
    x = torch.randn(n, generator=_gen(seed), dtype=torch.float32).to(torch.bfloat16)
    return x.view(torch.uint16).numpy() if hasattr(torch, "uint16") else \
        x.view(torch.int16).numpy().view(np.uint16)


def f32_uniform(n: int, seed: int = 2) -> np.ndarray:
    """n fp32 values uniform in [-1, 1)."""
    return (torch.rand(n, generator=_gen(seed), dtype=torch.float32) * 2 - 1).numpy()


def f16_bits_no_nan(n: int, seed: int = 3) -> np.ndarray:
    """n uniform fp16 bit patterns; a NaN encoding (exponent all ones, mantissa
    non-zero) has its exponent's second bit flipped, so none remain."""
    x = uint16_bits(n, seed).copy()
    nan = ((x & 0x7C00) == 0x7C00) & ((x & 0x03FF) != 0)
    x[nan] ^= 0x4000
    return x


def bank_patterns(n: int, width: int, seed: int = 5, smem_bytes: int = 228 * 1024,
                  aligned: bool = True) -> np.ndarray:
    """n warp access patterns of 32 byte addresses below smem_bytes.  With
    aligned=True every address is a multiple of the access width, as a real
    shared-memory access must be."""
    g = _gen(seed)
    units = smem_bytes // width if aligned else smem_bytes - width
    a = torch.randint(0, units, (n, 32), generator=g, dtype=torch.int64)
    if aligned:
        a = a * width
    return a.to(torch.int64).numpy().astype(np.uint32)


def active_masks(n: int, seed: int = 6) -> np.ndarray:
    """n random 32-bit lane masks."""
    b = random_bytes(4 * n, seed)
    return b.view(np.uint32).copy()
