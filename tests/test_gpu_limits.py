"""Parity at the API's limits: the most queries and requests one call takes,
the smallest and largest head_dim, and positions next to IS_MAX_POSITION
(where an overflowing segment is refused with IS_ST_POSITION and nothing of it
is written)."""
import numpy as np
import pytest

from synth import staging, workloads
from tests import gpu_helpers as gh
from tests import parity

pytestmark = pytest.mark.gpu

IS_MAX_QUERIES, IS_MAX_REQUESTS, IS_MAX_POSITION = 1024, 4096, 1 << 24


@pytest.fixture(scope="module")
def api():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api as a
    return a


def _spec(name, **kw):
    base = dict(num_layers=2, num_kv_heads=4, head_dim=64, kv_dtype="bf16",
                rope=workloads.RopeSpec(theta=1.0e4), n_users=16, facts_per_user=1100,
                length_dist=("uniform", 1, 7), emb_dim=128, emb_dtype="f16", n_queries=IS_MAX_QUERIES,
                k=16, query_kind="planted", start=("uniform", 0, 500), block_size=16, tokens_cap=16 * 7,
                block_layout="free_list", queries_share_user=True, seed=60)
    base.update(kw)
    return workloads.WorkloadSpec(name=name, **base)


@pytest.mark.parametrize("mode", ["per_query", "batched"])
def test_max_queries_in_one_call(api, mode):
    from kv_cache_injection_gb300 import _lib
    wl = workloads.generate(_spec("max_queries"))
    wl.users[:] = np.random.default_rng(1).integers(0, 16, size=IS_MAX_QUERIES).astype(np.int32)
    store = staging.load_store(wl, api)
    try:
        api.is_set_retrieval_mode(store, {"per_query": _lib.IS_RETRIEVAL_PER_QUERY,
                                          "batched": _lib.IS_RETRIEVAL_BATCHED}[mode])
        st = gh.check_fused_workload(api, wl, store, sample_tokens=400)
        assert st["tokens"] > IS_MAX_QUERIES * 16
    finally:
        store.destroy()


@pytest.mark.parametrize("head_dim,heads,dtype,style", [(16, 8, "f32", 0), (16, 8, "f32", 1),
                                                        (256, 2, "bf16", 1), (512, 2, "f16", 0),
                                                        (128, 4, "f32", 1)])
def test_head_dim_extremes(api, head_dim, heads, dtype, style):
    spec = _spec(f"d{head_dim}", head_dim=head_dim, num_kv_heads=heads, kv_dtype=dtype,
                 rope=workloads.RopeSpec(theta=5.0e5, style=style), n_users=3, facts_per_user=200,
                 n_queries=3, queries_share_user=False, emb_dtype="f32" if dtype == "f32" else "f16",
                 seed=61 + head_dim)
    wl = workloads.generate(spec)
    store = staging.load_store(wl, api)
    try:
        st = gh.check_fused_workload(api, wl, store, sample_tokens=200)
        assert st["tokens"] > 0
    finally:
        store.destroy()


@pytest.mark.parametrize("head_dim,dtype,style", [(512, "bf16", 1), (512, "f32", 0), (256, "f32", 1)])
def test_head_dim_beyond_the_kernels_is_refused(api, head_dim, dtype, style):
    """A head wider than 32 vectors per (half) head is refused before launch."""
    import torch
    spec = _spec("too_wide", head_dim=head_dim, num_kv_heads=1, kv_dtype=dtype,
                 rope=workloads.RopeSpec(theta=1.0e4, style=style), n_users=1, facts_per_user=20,
                 n_queries=1, queries_share_user=False, emb_dtype="f32" if dtype == "f32" else "f16", seed=64)
    wl = workloads.generate(spec)
    store = staging.load_store(wl, api)
    try:
        inp = staging.device_inputs(wl)
        cache = staging.canary_cache(wl)
        with pytest.raises(api.ISError) as e:
            gh.run_fused(api, store, wl, inp, cache)
        assert e.value.status == 8
        assert np.all(gh.changed_slots(cache, dtype) == False)   # noqa: E712
    finally:
        store.destroy()


def test_positions_next_to_the_limit(api):
    """Request 0 ends just below 2^24 and is injected exactly (the angle
    reduction holds at 16.7 M); request 1 would cross 2^24: it latches
    IS_ST_POSITION, gets segment length 0 and writes nothing."""
    import torch
    from kv_cache_injection_gb300 import _lib
    spec = _spec("near_max_pos", n_users=2, facts_per_user=300, n_queries=2, queries_share_user=False,
                 start=("uniform", IS_MAX_POSITION - 400, IS_MAX_POSITION - 300), k=16,
                 rope=workloads.LLAMA31_ROPE, seed=62)
    wl = workloads.generate(spec)
    store = staging.load_store(wl, api)
    try:
        inp = staging.device_inputs(wl)
        seg_start = inp["seg_start"].clone()
        seg_start[1] = IS_MAX_POSITION - 20
        inp["seg_start"] = seg_start
        cache = staging.canary_cache(wl)
        out = gh.run_fused(api, store, wl, inp, cache)
        assert out["status"] == _lib.IS_ST_POSITION
        assert out["seg_len"][1] == 0
        plans, lens = parity.oracle_plans(wl, out["ids"][:1])
        assert out["seg_len"][0] == lens[0] and int(wl.seg_start[0]) + lens[0] <= IS_MAX_POSITION
        want = np.array([e[3] for e in plans[0]], dtype=np.int64)
        assert np.array_equal(out["slot_map"][: len(want)], want)
        gh.assert_only_slots_changed(cache, "bf16", want)
        gk, gv = gh.gather_rows(cache, want)
        parity.compare_tokens(wl, gk, gv, plans[0], parity.oracle_freqs(wl), 0, parity.FactCache(wl))
    finally:
        store.destroy()


def test_max_requests_in_one_inject(api):
    """is_inject with IS_MAX_REQUESTS requests of 0 to 3 facts each."""
    import torch
    spec = _spec("max_requests", n_users=1, facts_per_user=3000, n_queries=IS_MAX_REQUESTS, k=3,
                 tokens_cap=3 * 7, start=("uniform", 0, 64), seed=63)
    wl = workloads.generate(spec)
    store = staging.load_store(wl, api, max_requests=IS_MAX_REQUESTS, max_queries=IS_MAX_QUERIES)
    try:
        rng = np.random.default_rng(2)
        R, stride = IS_MAX_REQUESTS, 3
        n_ids = rng.integers(0, 4, size=R).astype(np.int32)
        ids = np.full((R, stride), -3, dtype=np.int64)
        for r in range(R):
            ids[r, :n_ids[r]] = rng.choice(3000, size=n_ids[r], replace=False)
        inp = staging.device_inputs(wl)
        cache = staging.canary_cache(wl)
        seg_len = torch.empty(R, dtype=torch.int32, device="cuda")
        slot_map = torch.full((R * stride * 7,), -9, dtype=torch.int64, device="cuda")
        api.is_inject(store, torch.from_numpy(ids).cuda(), torch.from_numpy(n_ids).cuda(), inp["seg_start"],
                      staging.rope_params(wl, api), inp["block_table"],
                      api.make_cache_desc(16, wl.num_blocks, "bf16"), cache, users=inp["users"],
                      seg_len_out=seg_len, slot_mapping_out=slot_map)
        assert api.is_get_status(store) == 0
        rows = [ids[r, :n_ids[r]] for r in range(R)]
        plans, lens = parity.oracle_plans(wl, rows)
        assert np.array_equal(seg_len.cpu().numpy(), lens)
        want = np.concatenate([[e[3] for e in pl] for pl in plans]).astype(np.int64)
        assert np.array_equal(slot_map.cpu().numpy()[: len(want)], want)
        gh.assert_only_slots_changed(cache, "bf16", want)
        entries = [e for pl in plans for e in pl]
        pick = sorted(set(np.random.default_rng(3).choice(len(entries), 300, replace=False).tolist()))
        sample = [entries[i] for i in pick]
        gk, gv = gh.gather_rows(cache, [e[3] for e in sample])
        parity.compare_tokens(wl, gk, gv, sample, parity.oracle_freqs(wl), 0, parity.FactCache(wl))
    finally:
        store.destroy()
