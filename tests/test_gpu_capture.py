"""Context-Window Encoding capture through the C ABI.

A tiny multi-layer decoder (the oracle's, fp64, synthetic weights) encodes
each turn of a synthetic conversation together with its window of preceding
turns; its per-layer pre-RoPE K and V, rounded to bf16, stand in for the
engine's prefill output.  The library captures the facts' rows layer by layer;
injecting them must then equal the oracle's rotation of the captured K/V
(V bit-exact, K within 1 bf16 ulp), and a store built by is_store_add_facts
from the same fact rows must inject byte for byte the same cache.
"""
import numpy as np
import pytest

from oracle import cwe, model, numerics
from oracle import inject as oinject
from oracle import rope
from synth import staging
from tests import gpu_helpers as gh
from tests import parity

pytestmark = pytest.mark.gpu

L, D_MODEL, HQ, HK, D, E = 3, 64, 4, 2, 128, 64
BS = 16


@pytest.fixture(scope="module")
def api():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api as a
    return a


def _conversation(seed=0, n_turns=24, w=3):
    rng = np.random.default_rng(seed)
    m = model.make_model(rng, L, D_MODEL, HQ, HK, D, 2 * D_MODEL, theta=1.0e4, style=0)
    turns = [rng.standard_normal((int(n), D_MODEL)) for n in rng.integers(2, 11, size=n_turns)]
    windows, lengths, seqs = [], [], []
    for i in range(n_turns):
        wl, kv = cwe.encode_with_window(m, turns, i, w)
        windows.append(wl)
        lengths.append(len(turns[i]))
        seqs.append([(numerics.encode(k, "bf16"), numerics.encode(v, "bf16")) for k, v in kv])
    # layer buffers of the engine: every sequence back to back, [tokens][HK][D] bf16 bits
    layers = [(np.concatenate([s[l][0] for s in seqs]), np.concatenate([s[l][1] for s in seqs]))
              for l in range(L)]
    # the facts' own rows, [len][L][HK][D] per fact (what the store must hold)
    facts = [(np.stack([s[l][0][wl:] for l in range(L)], 1), np.stack([s[l][1][wl:] for l in range(L)], 1))
             for s, wl in zip(seqs, windows)]
    emb = rng.standard_normal((n_turns, E))
    emb = (emb / np.linalg.norm(emb, axis=1, keepdims=True)).astype(np.float16)
    return m, np.array(windows, np.int32), np.array(lengths, np.int32), layers, facts, emb


def _store(api, n, tokens, placement="device"):
    cfg = api.make_config(num_layers=L, num_kv_heads=HK, head_dim=D, emb_dim=E, kv_dtype="bf16",
                          emb_dtype="f16", max_facts=n, max_tokens=tokens, max_users=1, max_queries=4,
                          max_k=n, max_requests=4, kv_placement=placement)
    return api.is_store_create(cfg, 0)


def _to_dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _capture(api, store, windows, lengths, layers, emb, order=None):
    import torch
    api.is_store_capture_begin(store, 0, windows, lengths, torch.from_numpy(emb).cuda())
    for l in (order if order is not None else range(L)):
        api.is_store_capture_layer(store, l, _to_dev(layers[l][0]), _to_dev(layers[l][1]))
    return api.is_store_capture_end(store, len(lengths))


def _inject_all(api, store, n, lengths, start=5, seed=1):
    """Inject facts 0..n-1 in a shuffled order as one request; returns (cache, plan)."""
    import torch
    order = np.random.default_rng(seed).permutation(n)
    total = int(lengths.sum())
    n_blocks = (start + total) // BS + 2
    block_row = np.random.default_rng(seed + 1).permutation(n_blocks + 3)[:n_blocks].astype(np.int32)
    cache = torch.full((L, 2, n_blocks + 3, BS, HK, D), 0, dtype=torch.int16, device="cuda")
    cache.fill_(0x7FA5)
    cache = cache.view(torch.bfloat16)
    rope_p = api.make_rope(1.0e4, 0)
    cd = api.make_cache_desc(BS, n_blocks + 3, "bf16")
    ids = torch.from_numpy(order.astype(np.int64)[None]).cuda()
    n_ids = torch.tensor([n], dtype=torch.int32, device="cuda")
    seg_start = torch.tensor([start], dtype=torch.int32, device="cuda")
    bt = torch.from_numpy(block_row[None]).cuda()
    api.is_inject(store, ids, n_ids, seg_start, rope_p, bt, cd, cache)
    assert api.is_get_status(store) == 0
    plan, T = oinject.compose(order, lengths, start)
    slots = [oinject.slot(p, block_row, BS) for _, _, p in plan]
    return cache, plan, slots


@pytest.mark.parametrize("placement", ["device", "host"])
def test_capture_then_inject_matches_oracle(api, placement):
    m, windows, lengths, layers, facts, emb = _conversation()
    n, tokens = len(lengths), int(lengths.sum())
    store = _store(api, n, tokens, placement)
    try:
        ids = _capture(api, store, windows, lengths, layers, emb, order=[2, 0, 1])
        assert np.array_equal(ids, np.arange(n))
        assert api.is_store_info(store)["n_tokens"] == tokens
        cache, plan, slots = _inject_all(api, store, n, lengths)
        gk, gv = gh.gather_rows(cache, slots)
        freqs = rope.inv_freq(D, 1.0e4)
        for i, ((f, j, p), s) in enumerate(zip(plan, slots)):
            Kf, Vf = facts[f]
            assert np.array_equal(gv[i], Vf[j]), (f, j)
            o = oinject.rotated_key_rows(Kf[j], p, freqs, 0, "bf16")
            parity.check_rotated(gk[i], o, numerics.decode(Kf[j], "bf16"), 0, "bf16")
        gh.assert_only_slots_changed(cache, "bf16", slots)
    finally:
        store.destroy()


def test_capture_equals_add_facts_of_the_same_rows(api):
    import torch
    m, windows, lengths, layers, facts, emb = _conversation(seed=3, w=5)
    n, tokens = len(lengths), int(lengths.sum())
    a, b = _store(api, n, tokens), _store(api, n, tokens)
    try:
        _capture(api, a, windows, lengths, layers, emb)
        k = np.concatenate([f[0] for f in facts]).reshape(-1)
        v = np.concatenate([f[1] for f in facts]).reshape(-1)
        api.is_store_add_facts(b, 0, lengths, _to_dev(k), _to_dev(v), torch.from_numpy(emb).cuda())
        ca, _, _ = _inject_all(api, a, n, lengths, seed=7)
        cb, _, _ = _inject_all(api, b, n, lengths, seed=7)
        assert torch.equal(ca.view(torch.int16), cb.view(torch.int16))
        # retrieval sees the captured facts: a fact's own embedding ranks it first
        q = torch.from_numpy(emb[[11]]).cuda()
        users = torch.zeros(1, dtype=torch.int32, device="cuda")
        ids = torch.empty((1, 4), dtype=torch.int64, device="cuda")
        sc = torch.empty((1, 4), dtype=torch.float32, device="cuda")
        api.is_retrieve_topk(a, users, q, 4, ids, sc)
        assert int(ids[0, 0]) == 11
    finally:
        a.destroy()
        b.destroy()


def test_window_zero_capture_equals_independent_encoding(api):
    """w = 0: every window is empty, the captured rows are the independent
    encodings, and the layer buffers hold only fact tokens."""
    m, windows, lengths, layers, facts, emb = _conversation(seed=5, w=0)
    assert np.all(windows == 0)
    assert layers[0][0].shape[0] == lengths.sum()
    store = _store(api, len(lengths), int(lengths.sum()))
    try:
        _capture(api, store, windows, lengths, layers, emb)
        cache, plan, slots = _inject_all(api, store, len(lengths), lengths)
        gk, gv = gh.gather_rows(cache, slots)
        for i, ((f, j, p), s) in enumerate(zip(plan, slots)):
            assert np.array_equal(gv[i], facts[f][1][j])
    finally:
        store.destroy()


def test_capture_protocol_errors(api):
    import torch
    m, windows, lengths, layers, facts, emb = _conversation(seed=9, n_turns=6)
    n, tokens = len(lengths), int(lengths.sum())
    store = _store(api, n, tokens)
    try:
        k0, v0 = _to_dev(layers[0][0]), _to_dev(layers[0][1])
        with pytest.raises(api.ISError) as e:
            api.is_store_capture_layer(store, 0, k0, v0)          # nothing open
        assert e.value.status == 1
        api.is_store_capture_begin(store, 0, windows, lengths, torch.from_numpy(emb).cuda())
        with pytest.raises(api.ISError) as e:                        # second begin
            api.is_store_capture_begin(store, 0, windows, lengths, torch.from_numpy(emb).cuda())
        assert e.value.status == 1
        with pytest.raises(api.ISError) as e:                        # add_facts while open
            api.is_store_add_facts(store, 0, lengths[:1], k0, v0, torch.from_numpy(emb[:1]).cuda())
        assert e.value.status == 1
        api.is_store_capture_layer(store, 0, k0, v0)
        with pytest.raises(api.ISError) as e:                        # layer twice
            api.is_store_capture_layer(store, 0, k0, v0)
        assert e.value.status == 1
        with pytest.raises(api.ISError) as e:                        # layer out of range
            api.is_store_capture_layer(store, L, k0, v0)
        assert e.value.status == 4
        with pytest.raises(api.ISError) as e:                        # layers 1, 2 missing
            api.is_store_capture_end(store, n)
        assert e.value.status == 1
        info = api.is_store_info(store)
        assert info["n_facts"] == 0 and info["n_tokens"] == 0          # dropped
        with pytest.raises(ValueError):
            api.is_store_capture_begin(store, 0, windows[:2], lengths[:1], torch.from_numpy(emb).cuda())
        bad = lengths.copy()
        bad[2] = 0
        with pytest.raises(api.ISError) as e:
            api.is_store_capture_begin(store, 0, windows, bad, torch.from_numpy(emb).cuda())
        assert e.value.status == 1
        # abort, then a complete capture succeeds
        api.is_store_capture_begin(store, 0, windows, lengths, torch.from_numpy(emb).cuda())
        api.is_store_capture_abort(store)
        ids = _capture(api, store, windows, lengths, layers, emb)
        assert np.array_equal(ids, np.arange(n))
        assert api.is_store_info(store)["n_facts"] == n
    finally:
        store.destroy()


def test_large_capture_equals_add_facts():
    """A capture of 2000 facts (the fact search takes three 32-way rounds) with
    random windows stores exactly the fact rows: injecting all 2000 facts from
    it and from a store built by is_store_add_facts of the same rows gives the
    same cache byte for byte."""
    import torch
    gh.ensure_built()
    from kv_cache_injection_gb300 import api
    rng = np.random.default_rng(77)
    L, H, D, dt = 2, 4, 64, "bf16"
    tdt = staging.torch_dtype(dt)
    n = 2000
    lengths = rng.integers(1, 9, size=n).astype(np.int32)
    windows = rng.integers(0, 21, size=n).astype(np.int32)
    total = int((lengths + windows).sum())
    gen = torch.Generator(device="cuda").manual_seed(5)
    layers = [(torch.randn(total, H, D, device="cuda", generator=gen).to(tdt),
               torch.randn(total, H, D, device="cuda", generator=gen).to(tdt)) for _ in range(L)]
    emb = torch.nn.functional.normalize(torch.randn(n, 64, device="cuda", generator=gen), dim=1).half()

    def store():
        cfg = api.make_config(num_layers=L, num_kv_heads=H, head_dim=D, emb_dim=64, kv_dtype=dt,
                              emb_dtype="f16", max_facts=n, max_tokens=int(lengths.sum()), max_users=1,
                              max_queries=1, max_k=n // 2, max_requests=2)
        return api.is_store_create(cfg, 0)
    a, b = store(), store()
    try:
        api.is_store_capture_begin(a, 0, windows, lengths, emb)
        for l in range(L):
            api.is_store_capture_layer(a, l, layers[l][0], layers[l][1])
        assert np.array_equal(api.is_store_capture_end(a, n), np.arange(n))
        starts = np.cumsum(np.concatenate([[0], lengths + windows]))[:-1] + windows
        idx = torch.from_numpy(np.concatenate([np.arange(st, st + ln) for st, ln in zip(starts, lengths)])).cuda()
        k = torch.stack([layers[l][0].index_select(0, idx) for l in range(L)], 1).contiguous()
        v = torch.stack([layers[l][1].index_select(0, idx) for l in range(L)], 1).contiguous()
        api.is_store_add_facts(b, 0, lengths, k, v, emb)
        bs = 16
        order = rng.permutation(n).astype(np.int64).reshape(2, n // 2)
        seg = [int(lengths[order[r]].sum()) for r in range(2)]
        nbr = max(seg) // bs + 2
        nb = 2 * nbr
        bt = torch.arange(nb, dtype=torch.int32, device="cuda").reshape(2, nbr).flip(1).contiguous()
        rope = api.make_rope(1e4, 0)
        cd = api.make_cache_desc(bs, nb, dt)
        outs = []
        for st in (a, b):
            cache = torch.zeros((L, 2, nb, bs, H, D), dtype=tdt, device="cuda")
            api.is_inject(st, torch.from_numpy(order).cuda(), torch.full((2,), n // 2, dtype=torch.int32, device="cuda"),
                          torch.zeros(2, dtype=torch.int32, device="cuda"), rope, bt, cd, cache)
            assert api.is_get_status(st) == 0
            outs.append(cache)
        assert torch.equal(outs[0].view(torch.uint8), outs[1].view(torch.uint8))
        assert bool(outs[0].view(torch.int16).ne(0).any())
    finally:
        a.destroy()
        b.destroy()
