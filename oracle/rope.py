"""Rotary position embedding in fp64: frequencies and the per-pair rotation.

Chunked RoPE (InferScale, "Méthodologie", phase 2: "Stockage Pré-RoPE",
"Rotation Dynamique"; "방법론" Pre-RoPE 저장 / 동적 회전) stores each fact's keys
before the rotary embedding and, at serving time, applies the rotation of the
position each key takes in the composed segment.  Theorem 6 (same section,
"Garantie Théorique") states that this re-rotation is exact.  The pages do not
print the rotation; it is the RoFormer rotation (Su et al., 2021): dimension
pairs (a, b) are rotated by the angle p * inv_freq_i,

    a' = a cos(p w_i) - b sin(p w_i)
    b' = b cos(p w_i) + a sin(p w_i),      w_i = theta^(-2i/D),  i < D/2.

Pairing style 0 (NeoX, "rotate half") pairs dims (i, i + D/2); style 1 pairs
(2i, 2i + 1).  Values are never rotated.

Llama-3.1 frequency scaling (used by the Llama-3.1-8B workloads; not from the
pages) follows the published Llama 3.1 rule: with wavelength lam = 2 pi / w,
keep w if lam < L0 / high_freq_factor, use w / factor if lam > L0 /
low_freq_factor, and in between blend (1 - s) w / factor + s w with
s = (L0 / lam - low_freq_factor) / (high_freq_factor - low_freq_factor),
where L0 is the original context length.
"""
from __future__ import annotations

import math

import numpy as np


def inv_freq(head_dim: int, theta: float, scaling: int = 0, factor: float = 1.0,
             low_freq_factor: float = 1.0, high_freq_factor: float = 1.0,
             original_max_pos: int = 0) -> np.ndarray:
    """Rotation frequencies w_i, i = 0 .. D/2 - 1, in fp64."""
    if head_dim % 2:
        raise ValueError("head_dim must be even")
    out = np.empty(head_dim // 2, dtype=np.float64)
    for i in range(head_dim // 2):
        w = float(theta) ** (-(2.0 * i) / head_dim)
        if scaling == 1:
            lam = 2.0 * math.pi / w
            high_wavelen = original_max_pos / high_freq_factor
            low_wavelen = original_max_pos / low_freq_factor
            if lam < high_wavelen:
                pass
            elif lam > low_wavelen:
                w = w / factor
            else:
                s = (original_max_pos / lam - low_freq_factor) / (high_freq_factor - low_freq_factor)
                w = (1.0 - s) * w / factor + s * w
        elif scaling != 0:
            raise ValueError("unknown scaling")
        out[i] = w
    return out


def pair_indices(head_dim: int, style: int) -> tuple[np.ndarray, np.ndarray]:
    """Indices (first, second) of the D/2 rotated pairs; pair i uses frequency i."""
    half = head_dim // 2
    i = np.arange(half)
    if style == 0:
        return i, i + half
    if style == 1:
        return 2 * i, 2 * i + 1
    raise ValueError("unknown style")


def rotate(x: np.ndarray, position, freqs: np.ndarray, style: int) -> np.ndarray:
    """Rotate the last axis (head_dim) of x to ``position`` (scalar or array
    broadcasting against x.shape[:-1])."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    ia, ib = pair_indices(D, style)
    phi = np.asarray(position, dtype=np.float64)[..., None] * freqs     # [..., D/2]
    c, s = np.cos(phi), np.sin(phi)
    a, b = x[..., ia], x[..., ib]
    out = np.empty(np.broadcast_shapes(x.shape, phi.shape[:-1] + (D,)), dtype=np.float64)
    out[..., ia] = a * c - b * s
    out[..., ib] = b * c + a * s
    return out
