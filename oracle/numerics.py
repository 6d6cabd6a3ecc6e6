"""Storage encodings of the oracle: decode to fp64, round fp64 to storage.

The pages fix no precision; the workloads store K/V as fp32, bf16 or fp16
and embeddings as fp16 or fp32, and a paged cache may also hold FP8 E4M3
(the 8-bit cache format of vLLM, the engine the pages inject into).  bf16 is
held as uint16 bit patterns and E4M3 as uint8 (numpy has neither type).  Rounding to bf16 is round-to-nearest-even taken directly from the
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


E4M3_MAX = 448.0


def f64_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 to FP8 E4M3 (the OCP 8-bit format without infinities: 1 sign,
    4 exponent bits with bias 7, 3 stored significand bits; S.1111.111 is NaN),
    ties to even, saturating: magnitudes that round above 448 and infinities
    become +-448; NaN becomes 0x7F.  Returned as uint8 bits.

    A finite value is M * 2^q with an integer M of at most 4 bits; the quantum
    q is (exponent - 3) for normals (exponent >= -6) and 2^-9 below.
    """
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    a = np.minimum(np.abs(np.where(nan, 0.0, x)), 2.0 ** 20)
    _, e = np.frexp(a)                         # a in [2^(e-1), 2^e)
    q = np.maximum(e - 4, -9)
    M = np.rint(np.ldexp(a, -q))              # ties to even
    r = np.minimum(np.ldexp(M, q), E4M3_MAX)
    _, e2 = np.frexp(r)
    E = e2 - 1                                 # r in [2^E, 2^(E+1)) for r > 0
    normal = (r > 0) & (E >= -6)
    field = np.where(normal, E + 7, 0)
    mant = np.where(normal, np.ldexp(r, -E) * 8 - 8, np.ldexp(r, 9))
    bits = (field.astype(np.uint8) << np.uint8(3)) | np.rint(mant).astype(np.uint8)
    bits = bits | (np.signbit(x).astype(np.uint8) << np.uint8(7))
    return np.where(nan, np.uint8(0x7F), bits).astype(np.uint8)


def e4m3_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    field = (b >> 3) & 0xF
    mant = b & 0x7
    mag = np.where(field == 0, np.ldexp(mant.astype(np.float64), -9),
                   np.ldexp(1.0 + mant / 8.0, field - 7))
    return np.where((field == 15) & (mant == 7), np.nan, sign * mag)


def decode(arr: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f64(arr)
    if dtype == "e4m3":
        return e4m3_bits_to_f64(arr)
    if dtype in ("f32", "f16", "f64"):
        return np.asarray(arr).astype(np.float64)
    raise ValueError(dtype)


def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 -> storage encoding with round-to-nearest-even."""
    if dtype == "bf16":
        return f64_to_bf16_bits(x)
    if dtype == "e4m3":
        return f64_to_e4m3_bits(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "f16":
        return np.asarray(x, dtype=np.float64).astype(np.float16)
    if dtype == "f64":                          # exact cache, for the Theorem 3 check
        return np.asarray(x, dtype=np.float64)
    raise ValueError(dtype)


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the storage format at |x| (its unit in the last place)."""
    mant, emin = {"bf16": (7, -126), "f32": (23, -126), "f16": (10, -14), "e4m3": (3, -6)}[dtype]
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(a)                         # 2^(e-1) <= a < 2^e
    e = np.where(a > 0, e, emin + 1)           # zero: the subnormal spacing
    return np.ldexp(1.0, np.maximum(e - 1, emin) - mant)
