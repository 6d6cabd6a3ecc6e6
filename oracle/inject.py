"""Segment composition, slot mapping and the paged scatter-copy, in fp64.

InferScale ("Méthodologie", phase 2, "Rotation Dynamique" and "Injection";
"방법론" 동적 회전 / 주입): the retrieved facts are composed into one contiguous
segment, each stored pre-RoPE key is rotated to its new serving position, and
the composed K/V are scatter-copied into vLLM's paged KV cache; the engine then
prefills only the query tokens.

Readings where the pages are silent:
* the facts follow each other in the order given (descending score when they
  come from retrieval); token t of the segment (0-based) takes the absolute
  position p = start + t, and p is both the RoPE position and the logical cache
  index (vLLM convention);
* the paged cache is vLLM-style: physical block b holds block_size consecutive
  logical positions; ``slot(p) = block_table[p // bs] * bs + p % bs``; the cache
  is laid out [L][2][num_blocks][bs][H][D] with K at index 0 and V at 1;
* rotated keys are computed in fp64 and rounded to the cache type with
  round-to-nearest-even; values are copied bit for bit;
* every other element of the cache keeps its previous contents.

An FP8 E4M3 cache (vLLM's 8-bit KV cache; the pages do not treat it) stores
x / scale with one scale for K and one for V, rounded to nearest even and
saturated to +-448.  The division is taken as a multiplication by the
reciprocal rounded once to fp32, r = fp32(1 / scale) (equal to the division
for power-of-two scales such as vLLM's default 1.0).  The rotated key is
multiplied in fp64 like the rest of the rotation; for V, whose byte is a
quantised code of a stored value, the product fp32(v) * r is taken in fp32
as the kernel takes it, so both sides round the same number.
"""
from __future__ import annotations

import numpy as np

from . import numerics, rope


def compose(fact_ids, lengths, start: int):
    """Token plan of one request: list of (fact, t_in_fact, position) and the
    segment length."""
    plan = []
    t = 0
    for f in fact_ids:
        f = int(f)
        for j in range(int(lengths[f])):
            plan.append((f, j, start + t))
            t += 1
    return plan, t


def slot(position: int, block_row, block_size: int) -> int:
    return int(block_row[position // block_size]) * block_size + position % block_size


def rotated_key_rows(k_token: np.ndarray, position: int, freqs: np.ndarray, style: int,
                     kv_dtype: str) -> np.ndarray:
    """fp64 rotated keys of one token: k_token [L][H][D] in storage encoding."""
    return rope.rotate(numerics.decode(k_token, kv_dtype), position, freqs, style)


def scale_reciprocal(scale: float) -> np.float32:
    """fp32(1 / scale) of an fp32 scale, the reciprocal taken in fp64."""
    return np.float32(1.0 / float(np.float32(scale)))


def e4m3_key(k_rot: np.ndarray, k_scale: float) -> np.ndarray:
    """Rotated keys (fp64) into E4M3 bits: k * fp32(1 / k_scale), rounded once."""
    return numerics.f64_to_e4m3_bits(k_rot * float(scale_reciprocal(k_scale)))


def e4m3_value(v_enc: np.ndarray, kv_dtype: str, v_scale: float) -> np.ndarray:
    """Stored values into E4M3 bits: fp32(v) * fp32(1 / v_scale) in fp32, then
    rounded to E4M3 (bf16 and fp16 values are exact in fp32)."""
    v32 = numerics.decode(v_enc, kv_dtype).astype(np.float32)
    return numerics.f64_to_e4m3_bits((v32 * scale_reciprocal(v_scale)).astype(np.float64))


def inject(cache: np.ndarray, kv_dtype: str, fact_kv, fact_ids, lengths, start: int,
           block_row, block_size: int, freqs: np.ndarray, style: int, cache_dtype: str | None = None,
           k_scale: float = 1.0, v_scale: float = 1.0):
    """Scatter one request into ``cache`` (storage encoding, [L][2][NB][bs][H][D]),
    in place.  ``fact_kv(f)`` returns (K, V) of fact f as [len][L][H][D] in
    storage encoding.  ``cache_dtype`` "e4m3" selects an FP8 cache with the
    given scales; otherwise the cache has the store's type.  Returns (plan,
    seg_len, slots)."""
    plan, seg_len = compose(fact_ids, lengths, start)
    slots = []
    cur = None
    for f, j, p in plan:
        if cur is None or cur[0] != f:
            cur = (f,) + tuple(fact_kv(f))
        K, V = cur[1], cur[2]
        s = slot(p, block_row, block_size)
        slots.append(s)
        blk, off = divmod(s, block_size)
        k_rot = rotated_key_rows(K[j], p, freqs, style, kv_dtype)  # [L][H][D] fp64
        if cache_dtype == "e4m3":
            cache[:, 0, blk, off] = e4m3_key(k_rot, k_scale)
            cache[:, 1, blk, off] = e4m3_value(V[j], kv_dtype, v_scale)
        else:
            cache[:, 0, blk, off] = numerics.encode(k_rot, kv_dtype)
            cache[:, 1, blk, off] = V[j]
    return plan, seg_len, np.asarray(slots, dtype=np.int64)
