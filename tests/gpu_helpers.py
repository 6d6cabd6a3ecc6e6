"""GPU-side plumbing shared by the -m gpu tests (torch used as test plumbing)."""
from __future__ import annotations

import numpy as np

from synth import staging
from synth.workloads import CANARY_BITS
from tests import parity


def ensure_built():
    from kv_cache_injection_gb300 import build
    build.build()


def run_fused(api, store, wl, inp, cache, k=None, style=None, slot_cap=None, cache_dtype=None,
              k_scale=1.0, v_scale=1.0):
    import torch
    dev = cache.device
    Q = int(inp["users"].shape[0])
    k = wl.spec.k if k is None else k
    ids = torch.full((Q, k), -7, dtype=torch.int64, device=dev)
    scores = torch.zeros((Q, k), dtype=torch.float32, device=dev)
    seg_len = torch.full((Q,), -7, dtype=torch.int32, device=dev)
    cap = slot_cap or Q * k * int(wl.lengths.max())
    slot_map = torch.full((cap,), -9, dtype=torch.int64, device=dev)
    rope = staging.rope_params(wl, api, style)
    cdesc = api.make_cache_desc(wl.spec.block_size, cache.shape[2], cache_dtype or wl.spec.kv_dtype,
                                k_scale, v_scale)
    api.is_retrieve_and_inject(store, inp["users"], inp["q_emb"], k, inp["seg_start"], rope,
                               inp["block_table"], cdesc, cache, ids, scores, seg_len, slot_map)
    bits = api.is_get_status(store)
    torch.cuda.synchronize()
    return dict(ids=ids.cpu().numpy(), scores=scores.cpu().numpy(), seg_len=seg_len.cpu().numpy(),
                slot_map=slot_map.cpu().numpy(), status=bits)


def gather_rows(cache, slots):
    """Cache rows at the given slots: (K [n][L][H][D], V [n][L][H][D]) in storage encoding."""
    import torch
    L, _, NB, bs, H, D = cache.shape
    flat = cache.reshape(L, 2, NB * bs, H, D)
    idx = torch.as_tensor(np.asarray(slots, dtype=np.int64), device=cache.device)
    rows = flat.index_select(2, idx).permute(2, 0, 1, 3, 4).contiguous()   # [n][L][2][H][D]
    bits = staging.cache_bits(rows)
    return bits[:, :, 0], bits[:, :, 1]


def changed_slots(cache, dtype: str) -> np.ndarray:
    """bool [L][2][NB*bs]: which (layer, K/V, slot) rows differ from the canary."""
    import torch
    L, _, NB, bs, H, D = cache.shape
    if dtype == "f32":
        b = cache.view(torch.int32).reshape(L, 2, NB * bs, H * D)
    elif dtype == "e4m3":
        b = cache.reshape(L, 2, NB * bs, H * D)
    else:
        b = cache.view(torch.int16).reshape(L, 2, NB * bs, H * D)
    canary = CANARY_BITS[dtype]
    anydiff = (b != canary).any(-1)
    alldiff = (b != canary).all(-1)
    # a written row has no canary element left (every value is finite)
    assert torch.equal(anydiff, alldiff), "a cache row was partially written"
    return anydiff.cpu().numpy()


def assert_only_slots_changed(cache, dtype: str, slots) -> None:
    ch = changed_slots(cache, dtype)
    exp = np.zeros(ch.shape[2], dtype=bool)
    exp[np.asarray(slots, dtype=np.int64)] = True
    assert np.array_equal(ch, np.broadcast_to(exp, ch.shape)), \
        f"{int((ch != exp).sum())} cache rows differ from the expected set"


def check_fused_workload(api, wl, store, k=None, sample_tokens=160, seed=0, cache_dtype=None,
                         k_scale=1.0, v_scale=1.0):
    """Fused retrieve + inject of ``wl`` through ``store`` against the oracle:
    every top-k, segment length and slot; a sample of injected tokens; and
    that exactly the targeted cache rows changed.  Returns the cache too."""
    inp = staging.device_inputs(wl)
    cache = staging.canary_cache(wl, cache_dtype=cache_dtype)
    k = wl.spec.k if k is None else k
    out = run_fused(api, store, wl, inp, cache, k=k, cache_dtype=cache_dtype, k_scale=k_scale,
                    v_scale=v_scale)
    assert out["status"] == 0, hex(out["status"])
    swapped = 0
    for q in range(wl.spec.n_queries):
        o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, k)
        swapped += parity.check_topk(out["ids"][q], out["scores"][q], o_ids, o_sc, score_of, k)["swapped"]
    plans, lens = parity.oracle_plans(wl, out["ids"])
    assert np.array_equal(out["seg_len"], lens)
    want_slots = np.concatenate([[e[3] for e in pl] for pl in plans]).astype(np.int64)
    assert np.array_equal(out["slot_map"][: len(want_slots)], want_slots)
    assert len(np.unique(want_slots)) == len(want_slots)
    assert_only_slots_changed(cache, cache_dtype or wl.spec.kv_dtype, want_slots)
    # sampled tokens: first and last token of every segment, plus random ones
    entries = [e for pl in plans for e in pl]
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(len(entries), size=min(sample_tokens, len(entries)), replace=False).tolist())
    off = 0
    for pl in plans:
        if pl:
            pick.update([off, off + len(pl) - 1])
        off += len(pl)
    sample = [entries[i] for i in sorted(pick)]
    gk, gv = gather_rows(cache, [e[3] for e in sample])
    if cache_dtype == "e4m3":
        stats = parity.compare_tokens_fp8(wl, gk, gv, sample, parity.oracle_freqs(wl), wl.spec.rope.style,
                                          parity.FactCache(wl), k_scale, v_scale)
    else:
        stats = parity.compare_tokens(wl, gk, gv, sample, parity.oracle_freqs(wl), wl.spec.rope.style,
                                      parity.FactCache(wl))
    return {"tokens": int(lens.sum()), "swapped": swapped, "cache": cache, **stats}
