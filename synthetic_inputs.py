"""Seeded synthetic rank buffers for the virtual-rank collectives.

This module is the one piece shared by the oracle tests, the GPU parity tests
and the benchmark.  It only turns (seed, rank) into numbers; it holds none of
the collectives' arithmetic (no sums, no schedules, no rounding rules of the
method).

Generator: numpy's PCG64 bit generator, seeded with
``SeedSequence([seed, rank])`` so that every rank has its own stream and the
stream is the same on every platform numpy supports.  Raw 64-bit outputs are
mapped to values as follows:

* ``uniform_pm1_f32``: the top 24 bits k of each raw word give
  ``k * 2**-23 - 1`` -- uniform on [-1, 1) on a grid of 2**-23, every value
  exactly representable in fp32.
* ``normal_f32``: Box-Muller in float64 on two raw words
  (u1 in (0, 1], u2 in [0, 1)), scaled by sigma, cast to fp32.
* ``normal_bf16``: ``normal_f32`` converted to bf16 by torch (a library
  conversion, round to nearest even), returned as uint16 bit patterns.
* ``int32_bits``: the low 32 bits of each raw word.
* ``small_ints_f32``: integers in [-lim, lim] as fp32 (any summation order is
  exact while the partial sums stay below 2**24).

bf16 buffers are carried as ``numpy.uint16`` bit patterns everywhere on the
host side.
"""
from __future__ import annotations

import numpy as np

_BLOCK = 1 << 22  # values generated per numpy call, bounds temporary memory


def _bitgen(seed: int, rank: int) -> np.random.PCG64:
    return np.random.PCG64(np.random.SeedSequence([int(seed), int(rank)]))


def _raw(seed: int, rank: int, n: int) -> np.ndarray:
    return _bitgen(seed, rank).random_raw(int(n)).astype(np.uint64, copy=False)


def uniform_pm1_f32(seed: int, rank: int, n: int) -> np.ndarray:
    """Uniform[-1, 1) fp32 on a 2**-23 grid."""
    bg = _bitgen(seed, rank)
    out = np.empty(int(n), dtype=np.float32)
    for lo in range(0, int(n), _BLOCK):
        hi = min(int(n), lo + _BLOCK)
        k = (bg.random_raw(hi - lo) >> np.uint64(40)).astype(np.float64)
        out[lo:hi] = (k * (2.0 ** -23) - 1.0).astype(np.float32)
    return out


def normal_f32(seed: int, rank: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """N(0, sigma**2) fp32 by Box-Muller on pairs of raw words."""
    bg = _bitgen(seed, rank)
    out = np.empty(int(n), dtype=np.float32)
    for lo in range(0, int(n), _BLOCK):
        hi = min(int(n), lo + _BLOCK)
        r = bg.random_raw(2 * (hi - lo)).reshape(-1, 2)
        u1 = ((r[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u2 = (r[:, 1] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        out[lo:hi] = (z * sigma).astype(np.float32)
    return out


def f32_to_bf16_bits_library(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns via torch's conversion (input preparation only)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def normal_bf16(seed: int, rank: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """N(0, sigma**2) rounded to bf16, as uint16 bit patterns."""
    return f32_to_bf16_bits_library(normal_f32(seed, rank, n, sigma))


def uniform_pm1_bf16(seed: int, rank: int, n: int) -> np.ndarray:
    """Uniform[-1, 1) rounded to bf16, as uint16 bit patterns."""
    return f32_to_bf16_bits_library(uniform_pm1_f32(seed, rank, n))


def int32_bits(seed: int, rank: int, n: int) -> np.ndarray:
    """Uniformly random 32-bit patterns as int32."""
    bg = _bitgen(seed, rank)
    out = np.empty(int(n), dtype=np.int32)
    for lo in range(0, int(n), _BLOCK):
        hi = min(int(n), lo + _BLOCK)
        out[lo:hi] = (bg.random_raw(hi - lo) & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.int32)
    return out


def small_ints_f32(seed: int, rank: int, n: int, lim: int = 64) -> np.ndarray:
    """Integers in [-lim, lim] stored as fp32."""
    r = _raw(seed, rank, n)
    return ((r % np.uint64(2 * lim + 1)).astype(np.int64) - lim).astype(np.float32)


def small_ints_bf16(seed: int, rank: int, n: int, lim: int = 8) -> np.ndarray:
    """Integers in [-lim, lim] as bf16 bit patterns (exact in bf16 for lim <= 256)."""
    return f32_to_bf16_bits_library(small_ints_f32(seed, rank, n, lim))


def rank_buffers(kind: str, seed: int, nranks: int, n: int, **kw) -> list[np.ndarray]:
    """One buffer per virtual rank, each from its own (seed, rank) stream."""
    gen = {
        "uniform_f32": uniform_pm1_f32,
        "uniform_bf16": uniform_pm1_bf16,
        "normal_f32": normal_f32,
        "normal_bf16": normal_bf16,
        "int32_bits": int32_bits,
        "small_ints_f32": small_ints_f32,
        "small_ints_bf16": small_ints_bf16,
    }[kind]
    return [gen(seed, r, n, **kw) for r in range(nranks)]
