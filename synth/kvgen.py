"""Counter-based generator for synthetic pre-RoPE keys and raw values (host side).

Definition (shared, word for word, with ``synth/csrc/synthgen.cu``):

* ``mix(z)`` is the SplitMix64 output function (Steele, Lea & Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014):
  ``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
  z *= 0x94D049BB133111EB; z ^= z >> 31`` (all mod 2^64).
* A stream is keyed by ``base = mix((seed << 8) | stream)``; its n-th word is
  ``mix(base + (n + 1) * 0x9E3779B97F4A7C15)`` (the SplitMix64 sequence).
* Value ``i`` of a stream uses words ``3i, 3i+1, 3i+2``; their twelve 16-bit
  chunks ``u_j`` are summed, ``S = sum u_j``, and the value is
  ``z = (S - 393210) / 65536`` -- an Irwin-Hall approximation of N(0, 1)
  (mean 0, variance 1 - 2^-32) that is exact in fp32.
* The value is then rounded to the storage type: fp32 as is, bf16 and fp16
  with round-to-nearest-even.

Stream 0 holds keys, stream 1 values.  Within a stream, element
``(g, l, h, d)`` -- global token ``g`` of the workload's fact list, layer
``l``, KV head ``h``, dim ``d`` -- has index ``((g * L + l) * H + h) * D + d``.
"""
from __future__ import annotations

import numpy as np

M64 = (1 << 64) - 1
GAMMA = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

STREAM_K = 0
STREAM_V = 1


def mix(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    z = z ^ (z >> np.uint64(30))
    z = z * _C1
    z = z ^ (z >> np.uint64(27))
    z = z * _C2
    return z ^ (z >> np.uint64(31))


def stream_base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        return mix(np.array([((seed << 8) | stream) & M64], dtype=np.uint64))[0]


def words(base: np.uint64, n: np.ndarray) -> np.ndarray:
    n = np.asarray(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix(base + (n + np.uint64(1)) * GAMMA)


def irwin_hall_f32(seed: int, stream: int, index: np.ndarray) -> np.ndarray:
    """fp32 values for the given element indices of one stream."""
    index = np.asarray(index, dtype=np.uint64)
    base = stream_base(seed, stream)
    s = np.zeros(index.shape, dtype=np.int64)
    mask = np.uint64(0xFFFF)
    for j in range(3):
        w = words(base, index * np.uint64(3) + np.uint64(j))
        for c in range(4):
            s += ((w >> np.uint64(16 * c)) & mask).astype(np.int64)
    # |S - 393210| < 2^19, so the scaled value is exact in fp32.
    return ((s - 393210).astype(np.float64) / 65536.0).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); finite inputs only."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    return ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def encode(values_f32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return values_f32.astype(np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(values_f32)
    if dtype == "f16":
        return values_f32.astype(np.float16)
    raise ValueError(dtype)


def kv_elements(seed: int, stream: int, first: int, count: int, dtype: str,
                chunk: int = 1 << 22) -> np.ndarray:
    """Elements ``first .. first+count-1`` of one stream, in storage encoding
    (float32, uint16 bf16 bits or float16)."""
    out_dtype = {"f32": np.float32, "bf16": np.uint16, "f16": np.float16}[dtype]
    out = np.empty(count, dtype=out_dtype)
    for s in range(0, count, chunk):
        e = min(count, s + chunk)
        idx = np.arange(first + s, first + e, dtype=np.uint64)
        out[s:e] = encode(irwin_hall_f32(seed, stream, idx), dtype)
    return out
