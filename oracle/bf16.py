"""Storage-type conversions for the oracle (bf16 and fp32 caches).

bf16 is the upper half of an IEEE binary32: 1 sign bit, 8 exponent bits and 7
stored fraction bits (8 significant bits). A float64 value is rounded to bf16
*directly* (nearest, ties to even), never through float32 first, so there is no
double rounding. fp32 storage uses numpy's own float64 -> float32 rounding.
'f64' storage (no rounding at all) exists for the oracle's own exactness checks.
"""

from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> exact float64 values."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to bf16, nearest with ties to even; returns uint16 bits.

    A normal value x = m * 2**e (0.5 <= |m| < 1) keeps 8 significant bits, so it
    is rounded on the grid 2**(e-8); values below the smallest normal 2**-126 sit
    on the fixed subnormal grid 2**-133. Overflow gives +-inf, NaN gives a quiet NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    finite = np.isfinite(x)
    xf = np.where(finite, x, 0.0)
    m, e = np.frexp(xf)
    grid_exp = np.where(np.abs(xf) < 2.0 ** -126, -133, e - 8)
    step = np.ldexp(1.0, grid_exp)
    y = np.rint(xf / step) * step                      # rint: round half to even
    too_big = np.abs(y) > float(np.float32(3.3895313892515355e38))  # largest finite bf16
    y = np.where(too_big, np.copysign(np.inf, xf), y)
    y = np.where(finite, y, x)                         # inf and NaN pass through
    u = y.astype(np.float32).view(np.uint32)           # y is exactly representable in fp32
    bits = (u >> np.uint32(16)).astype(np.uint16)
    return np.where(np.isnan(x), np.uint16(0x7FC0), bits).astype(np.uint16)


def storage_to_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Stored cache/tensor values ('bf16' uint16 bits or 'f32' float32) -> float64."""
    if dtype == "bf16":
        return bf16_bits_to_f64(arr)
    if dtype == "f32":
        return np.asarray(arr, dtype=np.float32).astype(np.float64)
    if dtype == "f64":
        return np.asarray(arr, dtype=np.float64)
    raise ValueError(dtype)


def f64_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> storage representation, rounding to nearest even."""
    if dtype == "bf16":
        return f64_to_bf16_bits(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "f64":
        return np.array(x, dtype=np.float64, copy=True)
    raise ValueError(dtype)
