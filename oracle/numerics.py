"""Storage encodings of the oracle: decode to fp64, round fp64 to storage.

The pages fix no precision; the workloads store K/V as fp32 or bf16 and
embeddings as fp16 or fp32.  bf16 is held as uint16 bit patterns (numpy has no
bf16 type).  Rounding to bf16 is round-to-nearest-even taken directly from the
fp64 value (no intermediate fp32 rounding).
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):        # NaN patterns decode to NaN
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 to the nearest bf16 (ties to even), returned as uint16 bits.

    bf16 = 1 sign, 8 exponent, 7 stored significand bits.  A finite non-zero
    value is M * 2^q with an integer M of at most 8 bits; the quantum q is
    (exponent - 7) for normals and 2^-133 below the normal range.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                         # a = m * 2^e, m in [0.5, 1)
    q = np.maximum(e - 8, -133)
    M = np.rint(np.ldexp(a, -q))              # numpy rint: ties to even
    r = np.ldexp(M, q)
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    bits = (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    return bits | (np.signbit(x).astype(np.uint16) << np.uint16(15))


def decode(arr: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f64(arr)
    if dtype in ("f32", "f16", "f64"):
        return np.asarray(arr).astype(np.float64)
    raise ValueError(dtype)


def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 -> storage encoding with round-to-nearest-even."""
    if dtype == "bf16":
        return f64_to_bf16_bits(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "f16":
        return np.asarray(x, dtype=np.float64).astype(np.float16)
    if dtype == "f64":                          # exact cache, for the Theorem 3 check
        return np.asarray(x, dtype=np.float64)
    raise ValueError(dtype)


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the storage format at |x| (its unit in the last place)."""
    mant, emin = {"bf16": (7, -126), "f32": (23, -126), "f16": (10, -14)}[dtype]
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(a)                         # 2^(e-1) <= a < 2^e
    e = np.where(a > 0, e, emin + 1)           # zero: the subnormal spacing
    return np.ldexp(1.0, np.maximum(e - 1, emin) - mant)
