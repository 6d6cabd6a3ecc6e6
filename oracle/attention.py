"""A tiny one-layer causal decoder attention in fp64, for Theorems 3 and 6.

InferScale states two exactness results ("Contributions Clés" / "주요 기여"):

* Theorem 3: for causal decoder transformers, injecting precomputed KV states
  into the attention cache is exactly equivalent to injecting the same text into
  the prompt, provided the memory is injected at its intended positions;
* Theorem 6: re-rotating keys stored before RoPE to their serving positions is
  exact, so attention scores equal those of prefilling the facts there.

In a single layer a token's K and V depend only on its own hidden state, so the
equivalence is exact; with more layers it holds only for KV encoded in the joint
context (which is why the pages add Context-Window Encoding).  The checks
therefore use one layer.  Grouped-query attention: query head h reads KV head
h // (Hq / Hkv).
"""
from __future__ import annotations

import math

import numpy as np

from . import rope


def heads(x: np.ndarray, W: np.ndarray, n_heads: int) -> np.ndarray:
    """[T][d_model] @ [d_model][n_heads*D] -> [T][n_heads][D]."""
    y = np.asarray(x, dtype=np.float64) @ np.asarray(W, dtype=np.float64)
    return y.reshape(y.shape[0], n_heads, -1)


def causal_attention(q_rot, q_pos, k_rot, k_pos, v) -> np.ndarray:
    """out[i, h] = sum_{s: k_pos[s] <= q_pos[i]} softmax_s(<q_i, k_s>/sqrt(D)) v_s."""
    Tq, Hq, D = q_rot.shape
    Hk = k_rot.shape[1]
    group = Hq // Hk
    out = np.zeros((Tq, Hq, D), dtype=np.float64)
    for i in range(Tq):
        visible = np.asarray(k_pos) <= q_pos[i]
        for h in range(Hq):
            g = h // group
            logits = k_rot[visible, g, :] @ q_rot[i, h, :] / math.sqrt(D)
            w = np.exp(logits - logits.max())
            w /= w.sum()
            out[i, h] = w @ v[visible, g, :]
    return out


def prefill(x, positions, Wq, Wk, Wv, n_q_heads, n_kv_heads, freqs, style):
    """Full causal prefill of one sequence: returns (out, q_rot, k_rot, k_pre, v)."""
    q = heads(x, Wq, n_q_heads)
    k_pre = heads(x, Wk, n_kv_heads)
    v = heads(x, Wv, n_kv_heads)
    pos = np.asarray(positions)
    q_rot = rope.rotate(q, pos[:, None], freqs, style)
    k_rot = rope.rotate(k_pre, pos[:, None], freqs, style)
    return causal_attention(q_rot, pos, k_rot, pos, v), q_rot, k_rot, k_pre, v


def read_paged(cache: np.ndarray, block_row, block_size: int, ctx_len: int):
    """Gather logical positions 0 .. ctx_len-1 of one sequence from a one-layer
    paged cache [1][2][NB][bs][H][D]: returns (K [ctx][H][D], V [ctx][H][D])."""
    K = np.empty((ctx_len,) + cache.shape[4:], dtype=np.float64)
    V = np.empty_like(K)
    for p in range(ctx_len):
        blk, off = int(block_row[p // block_size]), p % block_size
        K[p] = cache[0, 0, blk, off]
        V[p] = cache[0, 1, blk, off]
    return K, V
