"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, small cases.

Sizes here finish on the oracle in seconds yet span several warps' work
items, several embedding tiles, ragged fact lists and partial cache blocks.
"""
import numpy as np
import pytest

from oracle import inject as oinject
from synth import kvgen, staging, workloads
from tests import gpu_helpers as gh
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api as a
    return a


@pytest.fixture(scope="module")
def tiny(api):
    wl = workloads.get("tiny")
    store = staging.load_store(wl, api)
    yield wl, store
    store.destroy()


def _full_compare(wl, cache, ids_rows, seg_len, slot_map, style):
    plans, lens = parity.oracle_plans(wl, ids_rows)
    assert np.array_equal(seg_len, lens)
    want_slots = np.concatenate([[e[3] for e in pl] for pl in plans]).astype(np.int64)
    assert np.array_equal(slot_map[: len(want_slots)], want_slots)
    facts = parity.FactCache(wl)
    freqs = parity.oracle_freqs(wl)
    entries = [e for pl in plans for e in pl]
    gk, gv = gh.gather_rows(cache, [e[3] for e in entries])
    stats = parity.compare_tokens(wl, gk, gv, entries, freqs, style, facts)
    gh.assert_only_slots_changed(cache, wl.spec.kv_dtype, want_slots)
    return stats


def test_device_generator_matches_host(api):
    import torch
    for dtype in ("f32", "bf16", "f16"):
        for first, n in [(0, 1000), (123456789, 4097), (2 ** 34 + 5, 333)]:
            t = torch.empty(n, dtype=staging.torch_dtype(dtype), device="cuda")
            staging.fill_kv(t, dtype, 9, 1, first)
            host = kvgen.kv_elements(9, 1, first, n, dtype)
            dev = staging.cache_bits(t)
            assert np.array_equal(dev.view(np.uint8), host.view(np.uint8)), dtype


@pytest.mark.parametrize("style", [0, 1])
def test_tiny_fused_full_cache(api, tiny, style):
    wl, store = tiny
    inp = staging.device_inputs(wl)
    cache = staging.canary_cache(wl)
    out = gh.run_fused(api, store, wl, inp, cache, style=style)
    assert out["status"] == 0
    o_ids, o_sc, score_of = parity.oracle_retrieve(wl, 0, wl.spec.k)
    parity.check_topk(out["ids"][0], out["scores"][0], o_ids, o_sc, score_of, wl.spec.k)
    _full_compare(wl, cache, out["ids"], out["seg_len"], out["slot_map"], style)


def test_tiny_topk_then_inject_equals_fused(api, tiny):
    import torch
    wl, store = tiny
    inp = staging.device_inputs(wl)
    k = wl.spec.k
    ids = torch.empty((1, k), dtype=torch.int64, device="cuda")
    sc = torch.empty((1, k), dtype=torch.float32, device="cuda")
    api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
    n_ids = (ids >= 0).sum(1).to(torch.int32)
    cache_a = staging.canary_cache(wl)
    rope = staging.rope_params(wl, api)
    cdesc = api.make_cache_desc(wl.spec.block_size, wl.num_blocks, wl.spec.kv_dtype)
    seg_len = torch.empty(1, dtype=torch.int32, device="cuda")
    api.is_inject(store, ids, n_ids, inp["seg_start"], rope, inp["block_table"], cdesc, cache_a,
                  users=inp["users"], seg_len_out=seg_len)
    assert api.is_get_status(store) == 0
    cache_b = staging.canary_cache(wl)
    out = gh.run_fused(api, store, wl, inp, cache_b)
    assert np.array_equal(out["ids"], ids.cpu().numpy())
    assert torch.equal(cache_a.view(torch.int32), cache_b.view(torch.int32))
    assert int(seg_len.item()) == int(out["seg_len"][0])


SMALL_BF16 = workloads.WorkloadSpec(
    name="small_bf16", num_layers=3, num_kv_heads=4, head_dim=64, kv_dtype="bf16",
    rope=workloads.RopeSpec(theta=1.0e4), n_users=5, facts_per_user=300,
    length_dist=("uniform", 1, 21), emb_dim=128, emb_dtype="f16", n_queries=5, k=9,
    query_kind="planted", start=("uniform", 0, 700), block_size=16, tokens_cap=9 * 21,
    block_layout="free_list", seed=11)


@pytest.mark.parametrize("dtype,style,scaled", [("bf16", 0, False), ("bf16", 1, False),
                                                ("f16", 0, True), ("f32", 0, False),
                                                ("f32", 1, True)])
def test_small_multi_user_fused(api, dtype, style, scaled):
    spec = SMALL_BF16.with_(kv_dtype=dtype, num_kv_heads=8 if dtype == "f32" else 4,
                            rope=workloads.RopeSpec(theta=5e5, style=style, scaling=1, factor=8.0,
                                                    low_freq_factor=1.0, high_freq_factor=4.0,
                                                    original_max_pos=64)
                            if scaled else workloads.RopeSpec(theta=1e4, style=style))
    wl = workloads.generate(spec)
    store = staging.load_store(wl, api)
    try:
        inp = staging.device_inputs(wl)
        cache = staging.canary_cache(wl)
        out = gh.run_fused(api, store, wl, inp, cache)
        assert out["status"] == 0
        for q in range(spec.n_queries):
            o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, spec.k)
            parity.check_topk(out["ids"][q], out["scores"][q], o_ids, o_sc, score_of, spec.k)
        _full_compare(wl, cache, out["ids"], out["seg_len"], out["slot_map"], style)
    finally:
        store.destroy()


def test_ragged_explicit_lists(api):
    """is_inject with ragged per-request fact lists (including an empty one),
    requests of different users, facts in arbitrary order."""
    import torch
    wl = workloads.generate(SMALL_BF16.with_(n_queries=5, seed=12))
    store = staging.load_store(wl, api)
    try:
        rng = np.random.default_rng(0)
        R, stride = 5, 9
        n_ids = np.array([9, 0, 1, 5, 7], dtype=np.int32)
        ids = np.full((R, stride), -5, dtype=np.int64)
        for r in range(R):
            facts = wl.user_facts(int(wl.users[r]))
            ids[r, :n_ids[r]] = rng.choice(facts, size=n_ids[r], replace=False)
        inp = staging.device_inputs(wl)
        cache = staging.canary_cache(wl)
        seg_len = torch.empty(R, dtype=torch.int32, device="cuda")
        slot_map = torch.full((int(R * stride * 21),), -9, dtype=torch.int64, device="cuda")
        rope = staging.rope_params(wl, api)
        cdesc = api.make_cache_desc(16, wl.num_blocks, "bf16")
        api.is_inject(store, torch.from_numpy(ids).cuda(), torch.from_numpy(n_ids).cuda(),
                      inp["seg_start"], rope, inp["block_table"], cdesc, cache, users=inp["users"],
                      seg_len_out=seg_len, slot_mapping_out=slot_map)
        assert api.is_get_status(store) == 0
        rows = [ids[r, :n_ids[r]] for r in range(R)]
        _full_compare(wl, cache, rows, seg_len.cpu().numpy(), slot_map.cpu().numpy(), 0)
    finally:
        store.destroy()


def test_ties_go_to_lower_fact_id(api):
    """Exactly tied scores (duplicated embeddings): lower fact ids win, including
    across the k-th boundary, and k up to the hard limit."""
    import torch
    spec = SMALL_BF16.with_(n_users=1, facts_per_user=1500, n_queries=3, k=1024, seed=13,
                            tokens_cap=1024 * 21, length_dist=("uniform", 1, 3))
    wl = workloads.generate(spec)
    base = wl.emb[:50].copy()
    wl.emb[:] = base[np.arange(1500) % 50]            # every embedding appears 30 times
    wl.queries[:] = base[[3, 17, 42]]
    store = staging.load_store(wl, api)
    try:
        inp = staging.device_inputs(wl)
        for k in (1, 29, 30, 31, 1024):
            ids = torch.empty((3, k), dtype=torch.int64, device="cuda")
            sc = torch.empty((3, k), dtype=torch.float32, device="cuda")
            api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
            g = ids.cpu().numpy()
            for q in range(3):
                o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, k)
                # every fact shares its score with 29 others: check the exact tie-break
                head = g[q][: min(k, 30)]
                assert np.array_equal(head, o_ids[: min(k, 30)]), (k, q)
                parity.check_topk(g[q], sc.cpu().numpy()[q], o_ids, o_sc, score_of, k)
        assert api.is_get_status(store) == 0
    finally:
        store.destroy()


def test_user_with_fewer_than_k_facts(api):
    import torch
    spec = SMALL_BF16.with_(n_users=2, facts_per_user=6, n_queries=2, k=9, seed=14)
    wl = workloads.generate(spec)
    store = staging.load_store(wl, api)
    try:
        inp = staging.device_inputs(wl)
        cache = staging.canary_cache(wl)
        out = gh.run_fused(api, store, wl, inp, cache)
        assert out["status"] == 0
        for q in range(2):
            o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, 9)
            assert len(o_ids) == 6
            parity.check_topk(out["ids"][q], out["scores"][q], o_ids, o_sc, score_of, 9)
        _full_compare(wl, cache, out["ids"], out["seg_len"], out["slot_map"], 0)
    finally:
        store.destroy()


def test_repeat_is_bit_identical(api, tiny):
    import torch
    wl, store = tiny
    inp = staging.device_inputs(wl)
    a = staging.canary_cache(wl)
    b = staging.canary_cache(wl)
    gh.run_fused(api, store, wl, inp, a)
    gh.run_fused(api, store, wl, inp, b)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_rope_frequencies_match_oracle(api):
    from oracle import rope
    r = workloads.LLAMA31_ROPE
    p = api.make_rope(r.theta, 0, 1, r.factor, r.low_freq_factor, r.high_freq_factor,
                      r.original_max_pos)
    got = api.is_rope_frequencies(p, 128)
    want = rope.inv_freq(128, r.theta, 1, r.factor, r.low_freq_factor, r.high_freq_factor,
                         r.original_max_pos)
    assert np.allclose(got, want, rtol=1e-14, atol=0)


@pytest.mark.parametrize("n", [1, 255, 2047, 2048, 2049])
def test_topk_around_the_register_path(api, n):
    """Users of n facts either side of 2048, where the top-k switches from bins
    counted by the similarity CTAs (kept zeroed between calls) to a shared-memory
    histogram.  Repeated calls with different k on one store, each against the
    oracle, and the fused path after them."""
    import torch
    spec = SMALL_BF16.with_(n_users=2, facts_per_user=n, n_queries=2, k=min(50, n), seed=40 + n,
                            length_dist=("uniform", 1, 3), tokens_cap=300 * 3)
    wl = workloads.generate(spec)
    store = staging.load_store(wl, api, max_k=300)
    try:
        inp = staging.device_inputs(wl)
        for k in (1, 50, 300, 7, 50):
            ids = torch.empty((2, k), dtype=torch.int64, device="cuda")
            sc = torch.empty((2, k), dtype=torch.float32, device="cuda")
            api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
            g, gs = ids.cpu().numpy(), sc.cpu().numpy()
            for q in range(2):
                o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, k)
                parity.check_topk(g[q], gs[q], o_ids, o_sc, score_of, k)
        cache = staging.canary_cache(wl)
        out = gh.run_fused(api, store, wl, inp, cache)
        assert out["status"] == 0
        for q in range(2):
            o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, wl.spec.k)
            parity.check_topk(out["ids"][q], out["scores"][q], o_ids, o_sc, score_of, wl.spec.k)
        _full_compare(wl, cache, out["ids"], out["seg_len"], out["slot_map"], 0)
        assert api.is_get_status(store) == 0
    finally:
        store.destroy()


def test_topk_heavy_ties_on_the_register_path(api):
    """2000 facts of one user whose embeddings take only 4 values: more than
    1024 rows share the k-th bin, so the exact radix select takes over from the
    bins the similarity CTAs counted; ties still go to the lower fact id."""
    import torch
    spec = SMALL_BF16.with_(n_users=1, facts_per_user=2000, n_queries=2, k=60, seed=61,
                            length_dist=("uniform", 1, 2), tokens_cap=60 * 2)
    wl = workloads.generate(spec)
    base = wl.emb[:4].copy()
    wl.emb[:] = base[np.arange(2000) % 4]
    wl.queries[:] = base[[1, 2]]
    store = staging.load_store(wl, api, max_k=1024)
    try:
        inp = staging.device_inputs(wl)
        for k in (60, 600, 1024):
            ids = torch.empty((2, k), dtype=torch.int64, device="cuda")
            sc = torch.empty((2, k), dtype=torch.float32, device="cuda")
            api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
            g = ids.cpu().numpy()
            for q in range(2):
                o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, k)
                head = min(k, 500)                    # the query's own value: 500 exact ties
                assert np.array_equal(g[q][:head], o_ids[:head]), (k, q)
                parity.check_topk(g[q], sc.cpu().numpy()[q], o_ids, o_sc, score_of, k)
        assert api.is_get_status(store) == 0
    finally:
        store.destroy()


@pytest.mark.parametrize("cache_dtype", [None, "e4m3"])
def test_chunk_pool_over_consecutive_launches(api, cache_dtype):
    """A launch with enough items per warp that the inject kernel hands half of
    them out through its claim counters (about 5600 tokens x 4 layers of 2 KiB
    rows), run three times: the counters alternate between launches, and every
    run must write the same cache, equal to the oracle's (an FP8 cache takes
    the even split instead)."""
    import torch
    spec = SMALL_BF16.with_(num_layers=4, num_kv_heads=8, head_dim=128, n_users=1, facts_per_user=400,
                            length_dist=("uniform", 24, 32), n_queries=1, k=200, tokens_cap=200 * 32,
                            seed=77)
    wl = workloads.generate(spec)
    store = staging.load_store(wl, api)
    try:
        inp = staging.device_inputs(wl)
        caches, outs = [], []
        for _ in range(3):
            c = staging.canary_cache(wl, cache_dtype=cache_dtype)
            outs.append(gh.run_fused(api, store, wl, inp, c, cache_dtype=cache_dtype))
            caches.append(c)
        assert all(o["status"] == 0 for o in outs)
        assert int(outs[0]["seg_len"][0]) * 4 >= 2 * 2432 * 4       # the pool is in use
        for c in caches[1:]:
            assert torch.equal(c.view(torch.uint8), caches[0].view(torch.uint8))
        if cache_dtype is None:
            _full_compare(wl, caches[0], outs[0]["ids"], outs[0]["seg_len"], outs[0]["slot_map"], 0)
        else:
            plans, lens = parity.oracle_plans(wl, outs[0]["ids"])
            want = np.concatenate([[e[3] for e in pl] for pl in plans]).astype(np.int64)
            gh.assert_only_slots_changed(caches[0], "e4m3", want)
    finally:
        store.destroy()


def test_host_buffer_call_equals_device_call(api):
    """is_retrieve_and_inject_host (host inputs and outputs, staged through the
    library's page-locked buffer) gives the device call's ids, scores, segment
    lengths and cache, on repeated calls and after its staging has grown: small
    inputs that the kernels read from the mapped buffer, inputs above 16 KiB
    (a block table padded by 1024 unused columns) that go over in one copy,
    then small inputs again."""
    import torch
    wl = workloads.generate(SMALL_BF16)
    s = wl.spec
    store = staging.load_store(wl, api)
    try:
        inp = staging.device_inputs(wl)
        dev_cache = staging.canary_cache(wl)
        out = gh.run_fused(api, store, wl, inp, dev_cache)
        assert out["status"] == 0
        rope = staging.rope_params(wl, api)
        cd = api.make_cache_desc(s.block_size, wl.num_blocks, s.kv_dtype)
        edt = np.float16 if s.emb_dtype == "f16" else np.float32
        users = np.ascontiguousarray(wl.users, dtype=np.int32)
        q = np.ascontiguousarray(wl.queries, dtype=edt)
        start = np.ascontiguousarray(wl.seg_start, dtype=np.int32)
        Q = len(users)
        bt0 = np.ascontiguousarray(wl.block_table, dtype=np.int32)
        padded = [np.ascontiguousarray(np.pad(bt0, ((0, 0), (0, p)))) for p in (64, 1024)]
        assert Q * padded[1].shape[1] * 4 > 16384
        for k, bt in ((s.k, bt0), (s.k, padded[0]), (s.k, padded[1]), (s.k, bt0)):
            host_cache = staging.canary_cache(wl)
            ids = np.full((Q, k), -5, dtype=np.int64)
            sc = np.zeros((Q, k), dtype=np.float32)
            ln = np.full(Q, -5, dtype=np.int32)
            api.is_retrieve_and_inject_host(store, users, q, k, start, rope, bt, cd, host_cache, ids, sc, ln)
            assert np.array_equal(ids, out["ids"])
            assert np.array_equal(sc.view(np.uint32), out["scores"].view(np.uint32))
            assert np.array_equal(ln, out["seg_len"])
            assert torch.equal(host_cache.view(torch.int16), dev_cache.view(torch.int16))
        assert api.is_get_status(store) == 0
        with pytest.raises(api.ISError):
            api.is_retrieve_and_inject_host(store, users, q, 0, start, rope, bt, cd, host_cache)
    finally:
        store.destroy()


def test_prepared_host_call_outputs_follow_each_call(api):
    """A prepared host call run back to back, with the rows of users and
    queries rotated between calls: each return hands back that call's ids,
    scores and segment lengths.  On the mapped path the calling thread
    returns on the completion word the inject kernel's last CTA writes, so
    the retrieval's outputs must be in the buffer by then; a stale buffer
    would return the previous rotation."""
    wl = workloads.generate(SMALL_BF16)
    s = wl.spec
    store = staging.load_store(wl, api)
    try:
        out = gh.run_fused(api, store, wl, staging.device_inputs(wl), staging.canary_cache(wl))
        assert out["status"] == 0
        rope = staging.rope_params(wl, api)
        cd = api.make_cache_desc(s.block_size, wl.num_blocks, s.kv_dtype)
        edt = np.float16 if s.emb_dtype == "f16" else np.float32
        Q, k = len(wl.users), s.k
        base_users = np.array(wl.users, dtype=np.int32)          # copies: the bound arrays are rewritten
        base_q = np.array(wl.queries, dtype=edt)
        users = base_users.copy()
        q = base_q.copy()
        start = np.ascontiguousarray(wl.seg_start, dtype=np.int32)
        bt = np.ascontiguousarray(wl.block_table, dtype=np.int32)
        ids = np.empty((Q, k), dtype=np.int64)
        sc = np.empty((Q, k), dtype=np.float32)
        ln = np.empty(Q, dtype=np.int32)
        call = api.prepare_retrieve_and_inject_host(store, users, q, k, start, rope, bt, cd,
                                                    staging.canary_cache(wl), ids, sc, ln)
        try:
            for i in range(16):
                r = (i * 3) % Q
                np.copyto(users, np.roll(base_users, r))
                np.copyto(q, np.roll(base_q, r, axis=0))
                ids.fill(-5)
                sc.fill(0.0)
                ln.fill(-5)
                call()
                assert np.array_equal(ids, np.roll(out["ids"], r, axis=0)), (i, r)
                assert np.array_equal(sc.view(np.uint32), np.roll(out["scores"], r, axis=0).view(np.uint32))
                assert np.array_equal(ln, np.roll(out["seg_len"], r)), (i, r)
        finally:
            call.close()
        assert api.is_get_status(store) == 0
    finally:
        store.destroy()


def test_host_call_with_nothing_to_inject(api):
    """Host-buffer calls whose inject launch has no token to move: a user
    without facts, then a user out of range.  Each call still returns (the
    inject kernel's last CTA writes the completion word with no work done)
    with the empty result and the cache untouched; the status bit comes only
    with the bad user; the call after them matches the device call."""
    import torch
    from kv_cache_injection_gb300 import _lib
    wl = workloads.generate(SMALL_BF16)
    s = wl.spec
    store = staging.load_store(wl, api, max_users=s.n_users + 1)      # the last user has no facts
    try:
        rope = staging.rope_params(wl, api)
        cd = api.make_cache_desc(s.block_size, wl.num_blocks, s.kv_dtype)
        edt = np.float16 if s.emb_dtype == "f16" else np.float32
        k = s.k
        q = np.array(wl.queries[:1], dtype=edt)
        start = np.array(wl.seg_start[:1], dtype=np.int32)
        bt = np.array(wl.block_table[:1], dtype=np.int32)
        for user, bits in ((s.n_users, 0), (s.n_users + 7, _lib.IS_ST_USER_RANGE)):
            cache = staging.canary_cache(wl)
            ids = np.full((1, k), 5, dtype=np.int64)
            sc = np.zeros((1, k), dtype=np.float32)
            ln = np.full(1, 5, dtype=np.int32)
            api.is_retrieve_and_inject_host(store, np.array([user], dtype=np.int32), q, k, start, rope, bt, cd,
                                            cache, ids, sc, ln)
            assert np.all(ids == -1) and np.all(np.isneginf(sc)) and ln[0] == 0, user
            assert torch.equal(cache.view(torch.int16), staging.canary_cache(wl).view(torch.int16))
            assert api.is_get_status(store) == bits, user
        inp = {"users": torch.tensor([int(wl.users[0])], dtype=torch.int32, device="cuda"),
               "q_emb": torch.from_numpy(q).cuda(), "seg_start": torch.from_numpy(start).cuda(),
               "block_table": torch.from_numpy(bt).cuda()}
        want_cache = staging.canary_cache(wl)
        want = gh.run_fused(api, store, wl, inp, want_cache)
        assert want["status"] == 0
        cache = staging.canary_cache(wl)
        ids = np.empty((1, k), dtype=np.int64)
        sc = np.empty((1, k), dtype=np.float32)
        ln = np.empty(1, dtype=np.int32)
        api.is_retrieve_and_inject_host(store, np.array([wl.users[0]], dtype=np.int32), q, k, start, rope, bt,
                                        cd, cache, ids, sc, ln)
        assert np.array_equal(ids, want["ids"]) and np.array_equal(ln, want["seg_len"])
        assert np.array_equal(sc.view(np.uint32), want["scores"].view(np.uint32))
        assert torch.equal(cache.view(torch.int16), want_cache.view(torch.int16))
    finally:
        store.destroy()


@pytest.mark.parametrize("n", [4096, 4097, 6000])
def test_per_query_topk_on_large_users(api, n):
    """The per-query retrieval kernel on users of 4096 facts (keys staged in
    shared memory) and more (keys read back from global memory), with the
    tensor-core path switched off, against the oracle for several k."""
    import torch
    from kv_cache_injection_gb300 import _lib
    spec = SMALL_BF16.with_(num_layers=1, n_users=2, facts_per_user=n, n_queries=2, k=50,
                            seed=90 + n % 7, length_dist=("uniform", 1, 2), tokens_cap=300 * 2)
    wl = workloads.generate(spec)
    store = staging.load_store(wl, api, max_k=300)
    try:
        api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_PER_QUERY)
        inp = staging.device_inputs(wl)
        for k in (1, 50, 300):
            ids = torch.empty((2, k), dtype=torch.int64, device="cuda")
            sc = torch.empty((2, k), dtype=torch.float32, device="cuda")
            api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
            g, gs = ids.cpu().numpy(), sc.cpu().numpy()
            for q in range(2):
                o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, k)
                parity.check_topk(g[q], gs[q], o_ids, o_sc, score_of, k)
        assert api.is_get_status(store) == 0
    finally:
        store.destroy()


def test_prepared_device_call_equals_direct_call(api, tiny):
    """api.prepare_retrieve_and_inject marshals once and reissues the call on
    the same buffers; after the inputs change in place, it must give what a
    direct call gives on the new inputs."""
    import torch
    wl, store = tiny
    s = wl.spec
    inp = staging.device_inputs(wl)
    Q, k = s.n_queries, s.k
    rope = staging.rope_params(wl, api)
    cd = api.make_cache_desc(s.block_size, wl.num_blocks, s.kv_dtype)
    outs = []
    for prepared in (True, False):
        cache = staging.canary_cache(wl)
        ids = torch.empty((Q, k), dtype=torch.int64, device="cuda")
        sc = torch.empty((Q, k), dtype=torch.float32, device="cuda")
        ln = torch.empty(Q, dtype=torch.int32, device="cuda")
        start = inp["seg_start"].clone()
        if prepared:
            call = api.prepare_retrieve_and_inject(store, inp["users"], inp["q_emb"], k, start, rope,
                                                   inp["block_table"], cd, cache, ids, sc, ln)
            call()
            start.add_(3)                              # new starts, same buffer
            staging.refill_canary(cache, s.kv_dtype)
            call()
        else:
            start.add_(3)
            api.is_retrieve_and_inject(store, inp["users"], inp["q_emb"], k, start, rope, inp["block_table"],
                                       cd, cache, ids, sc, ln)
        torch.cuda.synchronize()
        outs.append((ids.cpu(), ln.cpu(), cache.view(torch.int32).cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][2], outs[1][2])
    assert api.is_get_status(store) == 0
