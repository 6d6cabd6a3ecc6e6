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


class DeviceFactCache:
    """Whole facts' K and V (storage encoding, [len][L][H][D]) drawn by the
    device copy of the seeded input generator, which is bit-equal to
    ``synth.kvgen`` (``test_device_generator_matches_host``): the same inputs
    as ``parity.FactCache``, regenerated in milliseconds instead of seconds."""

    def __init__(self, wl):
        self.wl = wl
        self._m = {}

    def __call__(self, f: int):
        import torch
        from synth import kvgen
        f = int(f)
        if f not in self._m:
            s = self.wl.spec
            n = int(self.wl.lengths[f])
            first = int(self.wl.tok_base[f]) * s.token_elems
            out = []
            for stream in (kvgen.STREAM_K, kvgen.STREAM_V):
                t = torch.empty(n * s.token_elems, dtype=staging.torch_dtype(s.kv_dtype), device="cuda")
                staging.fill_kv(t, s.kv_dtype, s.seed, stream, first)
                out.append(staging.cache_bits(t).reshape(n, s.num_layers, s.num_kv_heads, s.head_dim))
            self._m[f] = tuple(out)
        return self._m[f]

    def token(self, f: int, t: int):
        K, V = self(f)
        return K[int(t)], V[int(t)]


def check_fused_workload(api, wl, store, k=None, sample_tokens=160, seed=0, cache_dtype=None,
                         k_scale=1.0, v_scale=1.0, all_tokens=False):
    """Fused retrieve + inject of ``wl`` through ``store`` against the oracle:
    every top-k, segment length and slot; the injected tokens; and that
    exactly the targeted cache rows changed.  ``all_tokens`` (True, or a list
    of query indices) compares every injected token of those queries, all
    layers and heads; the other queries' tokens are sampled (first and last of
    every segment plus ``sample_tokens`` random ones).  Returns the cache too."""
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
    full_q = (set(range(len(plans))) if all_tokens is True
              else set(int(q) for q in all_tokens) if all_tokens else set())
    freqs, style = parity.oracle_freqs(wl), wl.spec.rope.style
    stats = {"n": 0, "within_1ulp": 0, "floor_only": 0, "saturated": 0, "v_saturated": 0}
    # every token of the queries in full_q, one request at a time
    dfacts = DeviceFactCache(wl)
    n_full = 0
    for q in sorted(full_q):
        if not plans[q]:
            continue
        gk, gv = gather_rows(cache, [e[3] for e in plans[q]])
        st = parity.compare_runs(wl, gk, gv, plans[q], freqs, style, dfacts,
                                 (k_scale, v_scale) if cache_dtype == "e4m3" else None)
        for key, val in st.items():
            stats[key] += val
        n_full += len(plans[q])
    # the other queries: first and last token of every segment, plus random ones
    entries, ends = [], set()
    for q, pl in enumerate(plans):
        if q not in full_q:
            if pl:
                ends.update([len(entries), len(entries) + len(pl) - 1])
            entries.extend(pl)
    if entries:
        rng = np.random.default_rng(seed)
        pick = set(rng.choice(len(entries), size=min(sample_tokens, len(entries)), replace=False).tolist())
        sample = [entries[i] for i in sorted(pick | ends)]
        gk, gv = gather_rows(cache, [e[3] for e in sample])
        if cache_dtype == "e4m3":
            st = parity.compare_tokens_fp8(wl, gk, gv, sample, freqs, style, parity.FactCache(wl),
                                           k_scale, v_scale)
        else:
            st = parity.compare_tokens(wl, gk, gv, sample, freqs, style, parity.FactCache(wl))
        for key, val in st.items():
            stats[key] += val
    return {"tokens": int(lens.sum()), "tokens_compared_in_full": n_full, "swapped": swapped,
            "cache": cache, **stats}
