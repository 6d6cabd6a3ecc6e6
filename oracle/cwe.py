"""Context-Window Encoding of memory facts, in fp64.

Test infrastructure only, like the rest of ``oracle/``.

InferScale ("Méthodologie", phase 1, "Encodage de la Fenêtre de Contexte";
"방법론" 1. 오프라인 단계: 컨텍스트 윈도우 인코딩): encoding facts one by one loses
the context between them, so each memory fact is encoded together with a
configurable window of w preceding conversation turns, and only the target
fact's KV tensors are kept; the context tokens are dropped.  w = 0 is the
independent encoding.

Readings where the pages are silent:
* a conversation is a sequence of turns and each turn is one memory fact (its
  tokens are the fact's tokens); the window of turn i is turns max(0, i - w)
  .. i - 1, so turns near the start get shorter windows;
* the window and the fact are encoded as one sequence at positions 0, 1, ...;
  the stored keys are taken before RoPE, and every layer's attention depends
  only on relative positions (Theorem 6), so where the sequence starts does
  not change what is stored;
* stored per fact token and layer: the pre-RoPE key and the value, laid out
  [fact tokens][L][Hk][D] like the store's arena.
"""
from __future__ import annotations

import numpy as np

from . import model as tiny


def window_turns(i: int, w: int) -> range:
    return range(max(0, i - w), i)


def encode_with_window(m: tiny.TinyModel, turns, i: int, w: int, offset: int = 0):
    """Prefill of [window of turn i || turn i] at positions offset, offset + 1, ...

    Returns (window_len, kv) with kv[l] = (k_pre, v) over all tokens of the
    sequence (window first): the output an engine's prefill produces."""
    win = [turns[j] for j in window_turns(i, w)]
    x = np.concatenate(win + [turns[i]]) if win else np.asarray(turns[i])
    wl = sum(len(t) for t in win)
    _, kv = tiny.forward(m, x, np.arange(len(x)) + offset)
    return wl, kv


def capture(kv, window_len: int):
    """Keep the fact's tokens of one encoded sequence: ([n][L][Hk][D] K, same V)."""
    K = np.stack([k[window_len:] for k, _ in kv], axis=1)
    V = np.stack([v[window_len:] for _, v in kv], axis=1)
    return K, V


def cwe_fact_kv(m: tiny.TinyModel, turns, i: int, w: int, offset: int = 0):
    """Context-Window Encoding of turn i: its pre-RoPE K and V, [len][L][Hk][D]."""
    wl, kv = encode_with_window(m, turns, i, w, offset)
    return capture(kv, wl)
