"""A tiny multi-layer causal decoder in fp64: the offline encoder of the facts.

Test infrastructure only, like the rest of ``oracle/``.

InferScale precomputes each memory fact's KV by running the model over it
offline ("Méthodologie", phase 1) and intercepts the keys before RoPE
("Stockage Pré-RoPE").  The pages give no architecture and no weights; this is
the plain pre-norm decoder block of the Llama family with synthetic weights:

    a  = rmsnorm(h)             q, k, v = a Wq, a Wk, a Wv      (per head)
    h' = h + attn(RoPE(q), RoPE(k), v) Wo                       (causal, grouped-query)
    m  = rmsnorm(h')            h_next = h' + (silu(m W1) * (m W3)) W2

and each layer records k before its rotation and v.  ``past`` lets a sequence
attend to KV that is already in the cache (previous tokens or injected facts):
per layer the rotated keys, their positions and the values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import attention, rope


@dataclass
class TinyModel:
    layers: list                 # per layer: dict of Wq, Wk, Wv, Wo, W1, W2, W3
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_model: int
    freqs: np.ndarray
    style: int


def make_model(rng, n_layers: int, d_model: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
               d_ff: int, theta: float = 1.0e4, style: int = 0) -> TinyModel:
    """Synthetic weights, N(0, 1/fan_in) so activations stay O(1)."""
    def w(i, o):
        return rng.standard_normal((i, o)) / math.sqrt(i)
    layers = [dict(Wq=w(d_model, n_q_heads * head_dim), Wk=w(d_model, n_kv_heads * head_dim),
                   Wv=w(d_model, n_kv_heads * head_dim), Wo=w(n_q_heads * head_dim, d_model),
                   W1=w(d_model, d_ff), W3=w(d_model, d_ff), W2=w(d_ff, d_model))
              for _ in range(n_layers)]
    return TinyModel(layers, n_q_heads, n_kv_heads, head_dim, d_model,
                     rope.inv_freq(head_dim, theta), style)


def rmsnorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def forward(model: TinyModel, x: np.ndarray, positions, past=None):
    """Prefill of tokens x [T][d_model] at ``positions`` after ``past``.

    Returns (h_out [T][d_model], kv) with kv[l] = (k_pre [T][Hk][D], v [T][Hk][D]).
    ``past[l]`` = (k_rot [S][Hk][D], pos [S], v [S][Hk][D]) or None."""
    h = np.asarray(x, dtype=np.float64)
    pos = np.asarray(positions)
    kv = []
    for l, W in enumerate(model.layers):
        a = rmsnorm(h)
        q = attention.heads(a, W["Wq"], model.n_q_heads)
        k_pre = attention.heads(a, W["Wk"], model.n_kv_heads)
        v = attention.heads(a, W["Wv"], model.n_kv_heads)
        q_rot = rope.rotate(q, pos[:, None], model.freqs, model.style)
        k_rot = rope.rotate(k_pre, pos[:, None], model.freqs, model.style)
        if past is not None and past[l] is not None:
            pk, ppos, pv = past[l]
            k_all = np.concatenate([pk, k_rot])
            pos_all = np.concatenate([np.asarray(ppos), pos])
            v_all = np.concatenate([pv, v])
        else:
            k_all, pos_all, v_all = k_rot, pos, v
        o = attention.causal_attention(q_rot, pos, k_all, pos_all, v_all)
        h = h + o.reshape(o.shape[0], -1) @ W["Wo"]
        m = rmsnorm(h)
        h = h + (silu(m @ W["W1"]) * (m @ W["W3"])) @ W["W2"]
        kv.append((k_pre, v))
    return h, kv
