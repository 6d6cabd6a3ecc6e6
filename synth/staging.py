"""Device-side staging of a synthetic workload.

Fills pre-RoPE K and raw V on the GPU with the counter-based generator
(``libsynthgen.so``, same definition as ``synth.kvgen``), uploads embeddings,
queries and block tables, and hands the facts to a store through the public
``is_store_add_facts`` call, a few hundred MB at a time.  Input plumbing only.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import kvgen
from .workloads import CANARY_BITS, Workload, cache_shape

_HERE = os.path.dirname(os.path.abspath(__file__))
SYNTH_LIB = os.path.join(_HERE, "lib", "libsynthgen.so")
DTYPE_CODE = {"f32": 0, "bf16": 1, "f16": 2}
_synth = None


def _lib():
    global _synth
    if _synth is None:
        if not os.path.exists(SYNTH_LIB):
            raise RuntimeError(f"{SYNTH_LIB} missing: run kv_cache_injection_gb300.build.build()")
        lib = ctypes.CDLL(SYNTH_LIB)
        lib.synth_fill_kv.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_int,
                                      ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p]
        lib.synth_fill_kv.restype = ctypes.c_int
        _synth = lib
    return _synth


def torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "e4m3": torch.uint8}[dtype]


def fill_kv(out, dtype: str, seed: int, stream_id: int, first: int) -> None:
    """Fill ``out`` (contiguous CUDA tensor) with elements first.. of one stream."""
    import torch
    rc = _lib().synth_fill_kv(out.data_ptr(), DTYPE_CODE[dtype], seed, stream_id, first,
                              out.numel(), torch.cuda.current_stream().cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_kv failed ({rc})")


def store_config(wl: Workload, api, **overrides):
    s = wl.spec
    kw = dict(num_layers=s.num_layers, num_kv_heads=s.num_kv_heads, head_dim=s.head_dim,
              emb_dim=s.emb_dim, kv_dtype=s.kv_dtype, emb_dtype=s.emb_dtype,
              max_facts=s.n_facts, max_tokens=wl.total_tokens, max_users=s.n_users,
              max_queries=max(s.n_queries, 1), max_k=max(s.k, 1),
              max_requests=max(s.n_queries, 1), max_facts_per_user=s.facts_per_user)
    kw.update(overrides)
    return api.make_config(**kw)


def rope_params(wl: Workload, api, style: int | None = None):
    r = wl.spec.rope
    return api.make_rope(r.theta, r.style if style is None else style, r.scaling, r.factor,
                         r.low_freq_factor, r.high_freq_factor, r.original_max_pos)


def load_store(wl: Workload, api, device: int = 0, chunk_bytes: int = 1 << 30, **cfg_overrides):
    """Create a store sized for ``wl`` and add every fact, user by user."""
    import torch
    s = wl.spec
    store = api.is_store_create(store_config(wl, api, **cfg_overrides), device)
    tdt = torch_dtype(s.kv_dtype)
    per_tok = s.token_elems
    max_tok = max(int(chunk_bytes // (per_tok * s.elt_bytes)), int(wl.lengths.max()))
    kbuf = torch.empty(max_tok * per_tok, dtype=tdt, device=f"cuda:{device}")
    vbuf = torch.empty_like(kbuf)
    edt = torch.float16 if s.emb_dtype == "f16" else torch.float32
    for u in range(s.n_users):
        facts = wl.user_facts(u)
        i = 0
        while i < len(facts):
            j, tok = i, 0
            while j < len(facts) and tok + int(wl.lengths[facts[j]]) <= max_tok:
                tok += int(wl.lengths[facts[j]])
                j += 1
            f0 = int(facts[i])
            first = int(wl.tok_base[f0]) * per_tok
            k = kbuf[: tok * per_tok]
            v = vbuf[: tok * per_tok]
            fill_kv(k, s.kv_dtype, s.seed, kvgen.STREAM_K, first)
            fill_kv(v, s.kv_dtype, s.seed, kvgen.STREAM_V, first)
            emb = torch.from_numpy(np.ascontiguousarray(wl.emb[facts[i:j]])).to(edt).to(k.device)
            ids = api.is_store_add_facts(store, u, wl.lengths[facts[i:j]], k, v, emb)
            assert np.array_equal(ids, facts[i:j]), "store ids must follow generator order"
            i = j
    del kbuf, vbuf
    return store


def device_inputs(wl: Workload, device: int = 0) -> dict:
    import torch
    dev = f"cuda:{device}"
    edt = torch.float16 if wl.spec.emb_dtype == "f16" else torch.float32
    return dict(users=torch.from_numpy(wl.users).to(dev),
                q_emb=torch.from_numpy(np.ascontiguousarray(wl.queries)).to(edt).to(dev),
                seg_start=torch.from_numpy(wl.seg_start).to(dev),
                block_table=torch.from_numpy(np.ascontiguousarray(wl.block_table)).to(dev))


def canary_cache(wl: Workload, device: int = 0, num_blocks: int | None = None,
                 cache_dtype: str | None = None):
    """A paged cache for ``wl`` filled with the canary; ``cache_dtype`` "e4m3"
    gives an FP8 cache (uint8 elements), else the store's type."""
    import torch
    s = wl.spec
    dt = cache_dtype or s.kv_dtype
    shape = cache_shape(s, wl.num_blocks if num_blocks is None else num_blocks)
    cache = torch.empty(shape, dtype=torch_dtype(dt), device=f"cuda:{device}")
    refill_canary(cache, dt)
    return cache


def refill_canary(cache, dtype: str) -> None:
    import torch
    if dtype == "f32":
        cache.view(torch.int32).fill_(CANARY_BITS["f32"])
    elif dtype == "e4m3":
        cache.fill_(CANARY_BITS["e4m3"])
    else:
        cache.view(torch.int16).fill_(CANARY_BITS[dtype])


def cache_bits(cache) -> np.ndarray:
    """Host copy in storage encoding: float32, float16, uint16 bits for bf16,
    uint8 bits for an FP8 cache."""
    import torch
    if cache.dtype in (torch.float32, torch.uint8):
        return cache.cpu().numpy()
    bits = cache.view(torch.int16).cpu().numpy().view(np.uint16)
    return bits.view(np.float16) if cache.dtype == torch.float16 else bits
