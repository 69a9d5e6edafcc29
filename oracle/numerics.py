"""Lane arithmetic of the oracle.

The pages fix the data types (FP32 / FP16 / BF16 and the SUM / MAX / MIN ops
of ``hccl_allreduce``, [hccl article] section "hccl_allreduce接口详解") and the
benchmark fixes the precision: fp32 sums, bf16 inputs accumulated in fp32 and
rounded once, int32 sums.  So the oracle computes:

* fp32: numpy float32 addition, one IEEE binary32 round-to-nearest-even per
  add, in exactly the association the simulated schedule produces;
* int32: addition modulo 2**32 (carried as uint32, which wraps);
* bf16: widened exactly to fp32 (a bf16 is the upper half of a binary32),
  accumulated as fp32, rounded once to bf16, round to nearest, ties to even,
  written here from the bit layout.  NaN stays a quiet NaN with its sign.

bf16 values are carried as uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np

DTYPES = ("f32", "bf16", "i32", "f16")
ESIZE = {"f32": 4, "bf16": 2, "i32": 4, "f16": 2}  # bytes per stored element
ACC_ESIZE = {"f32": 4, "bf16": 4, "i32": 4, "f16": 4}  # bytes per accumulated element
OPS = ("sum", "max", "min")


def storage_dtype(dtype: str):
    return {"f32": np.float32, "bf16": np.uint16, "i32": np.int32, "f16": np.float16}[dtype]


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening: place the 16 bits in the upper half of a binary32."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """binary32 -> bf16 bits, round to nearest, ties to even.

    With u the 32 bits of x, the kept part is u >> 16 and the dropped part is
    u & 0xFFFF.  Adding 0x7FFF plus the kept part's lowest bit rounds up
    exactly when the dropped part is above one half, or equal to one half with
    an odd kept part; a carry out of the mantissa moves into the exponent
    (the largest finite values round to infinity, as the format requires).
    NaN inputs keep their sign and top payload bits and get the quiet bit set.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    is_nan = (u & np.uint64(0x7FFFFFFF)) > np.uint64(0x7F800000)
    if np.any(is_nan):
        quiet = ((u >> np.uint64(16)) | np.uint64(0x0040)).astype(np.uint16)
        rounded = np.where(is_nan, quiet, rounded)
    return rounded


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Stored values -> accumulation lane type (a fresh array).  fp16 is
    widened by numpy's binary16 -> binary32 conversion (exact)."""
    if dtype == "f32":
        return np.array(x, dtype=np.float32, copy=True)
    if dtype == "f16":
        return np.asarray(x, dtype=np.float16).astype(np.float32)
    if dtype == "bf16":
        return bf16_to_f32(x).copy()
    if dtype == "i32":
        return np.array(x, dtype=np.int32).view(np.uint32).copy()
    raise ValueError(dtype)


def narrow(acc: np.ndarray, dtype: str) -> np.ndarray:
    """Accumulation lane type -> stored values (one rounding for bf16 and
    fp16; fp16 by numpy's binary32 -> binary16 conversion, round to nearest
    even)."""
    if dtype == "f32":
        return np.array(acc, dtype=np.float32, copy=True)
    if dtype == "f16":
        with np.errstate(over="ignore"):
            return np.asarray(acc, dtype=np.float32).astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16(acc)
    if dtype == "i32":
        return np.array(acc, dtype=np.uint32).view(np.int32).copy()
    raise ValueError(dtype)


def add(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """One elementwise add in the lane type (fp32 RNE, or uint32 wrap)."""
    assert a.dtype == b.dtype and a.dtype in (np.float32, np.uint32), (a.dtype, b.dtype)
    with np.errstate(over="ignore", invalid="ignore"):
        return a + b


def combine(a: np.ndarray, b: np.ndarray, op: str) -> np.ndarray:
    """One reduction step a (+) b in the lane type.

    sum: ``add``.  max / min (the hccl article lists SUM, MAX and MIN; it does
    not say how NaN or signed zeros behave): the reading taken is
    max(a, b) = b if b > a or a is NaN, else a (and min with b < a).  A NaN
    operand is passed over while a number is present, and of two equal
    values (+0 and -0) the first is kept, so the result depends on the
    association only through the sign of zero and NaN payloads.  int32
    compares as signed."""
    if op == "sum":
        return add(a, b)
    assert a.dtype == b.dtype
    if a.dtype == np.uint32:
        ai, bi = a.view(np.int32), b.view(np.int32)
        take_b = bi > ai if op == "max" else bi < ai
    else:
        with np.errstate(invalid="ignore"):
            take_b = ((b > a) if op == "max" else (b < a)) | np.isnan(a)
    return np.where(take_b, b, a)


def same_bits(a: np.ndarray, b: np.ndarray) -> bool:
    """Bitwise equality of two stored buffers."""
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    if a.shape != b.shape or a.dtype.itemsize != b.dtype.itemsize:
        return False
    return bool(np.array_equal(a.view(np.uint8), b.view(np.uint8)))
