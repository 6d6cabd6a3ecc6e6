"""The batched (tensor-core) retrieval path against the oracle and against the
per-query path: queries grouped by user, more than 64 queries of one user
(two groups), users with few queries, an unknown user, and the fused
retrieve + inject on top of it."""
import numpy as np
import pytest

from synth import staging, workloads
from tests import gpu_helpers as gh
from tests import parity

pytestmark = pytest.mark.gpu

MIX = workloads.WorkloadSpec(
    name="batched_mix", num_layers=2, num_kv_heads=4, head_dim=64, kv_dtype="bf16",
    rope=workloads.RopeSpec(theta=1.0e4), n_users=3, facts_per_user=700,
    length_dist=("uniform", 1, 9), emb_dim=192, emb_dtype="f16", n_queries=100, k=16,
    query_kind="planted", start=("uniform", 0, 300), block_size=16, tokens_cap=16 * 9,
    block_layout="free_list", queries_share_user=True, seed=41)


@pytest.fixture(scope="module")
def env():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api
    wl = workloads.generate(MIX)
    # 70 queries of user 0 (two groups), 20 of user 1, 10 of user 2, interleaved
    users = np.array([0] * 70 + [1] * 20 + [2] * 10, dtype=np.int32)
    wl.users[:] = np.random.default_rng(0).permutation(users)
    store = staging.load_store(wl, api)
    yield api, wl, store
    store.destroy()


def _retrieve(api, store, wl, users=None):
    import torch
    inp = staging.device_inputs(wl)
    Q, k = wl.spec.n_queries, wl.spec.k
    u = inp["users"] if users is None else torch.from_numpy(users).cuda()
    ids = torch.full((Q, k), -7, dtype=torch.int64, device="cuda")
    sc = torch.zeros((Q, k), dtype=torch.float32, device="cuda")
    api.is_retrieve_topk(store, u, inp["q_emb"], k, ids, sc)
    bits = api.is_get_status(store)
    return ids.cpu().numpy(), sc.cpu().numpy(), bits


def test_batched_topk_matches_oracle(env):
    from kv_cache_injection_gb300 import _lib
    api, wl, store = env
    api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_BATCHED)
    try:
        ids, sc, bits = _retrieve(api, store, wl)
    finally:
        api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_AUTO)
    assert bits == 0
    for q in range(wl.spec.n_queries):
        o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, wl.spec.k)
        parity.check_topk(ids[q], sc[q], o_ids, o_sc, score_of, wl.spec.k)


def test_batched_equals_per_query(env):
    from kv_cache_injection_gb300 import _lib
    api, wl, store = env
    api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_BATCHED)
    try:
        ids_b, sc_b, _ = _retrieve(api, store, wl)
    finally:
        api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_PER_QUERY)
    try:
        ids_p, sc_p, _ = _retrieve(api, store, wl)
    finally:
        api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_AUTO)
    assert np.max(np.abs(sc_b - sc_p)) <= 2e-6
    # ids may differ only between scores closer than the accumulation-order noise
    diff = ids_b != ids_p
    for q, r in zip(*np.nonzero(diff)):
        assert abs(sc_p[q, r] - sc_b[q, r]) <= 2e-6


def test_batched_unknown_user(env):
    from kv_cache_injection_gb300 import _lib
    api, wl, store = env
    users = wl.users.copy()
    users[5] = 9
    api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_BATCHED)
    try:
        ids, sc, bits = _retrieve(api, store, wl, users)
    finally:
        api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_AUTO)
    assert bits == _lib.IS_ST_USER_RANGE
    assert np.all(ids[5] == -1)
    o_ids, o_sc, score_of = parity.oracle_retrieve(wl, 6, wl.spec.k)
    parity.check_topk(ids[6], sc[6], o_ids, o_sc, score_of, wl.spec.k)


def test_batched_fused_inject(env):
    from kv_cache_injection_gb300 import _lib
    api, wl, store = env
    inp = staging.device_inputs(wl)
    cache = staging.canary_cache(wl)
    api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_BATCHED)
    try:
        out = gh.run_fused(api, store, wl, inp, cache)
    finally:
        api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_AUTO)
    assert out["status"] == 0
    plans, lens = parity.oracle_plans(wl, out["ids"])
    assert np.array_equal(out["seg_len"], lens)
    want = np.concatenate([[e[3] for e in pl] for pl in plans]).astype(np.int64)
    assert np.array_equal(out["slot_map"][: len(want)], want)
    gh.assert_only_slots_changed(cache, "bf16", want)
    entries = [e for pl in plans for e in pl][::7]
    gk, gv = gh.gather_rows(cache, [e[3] for e in entries])
    parity.compare_tokens(wl, gk, gv, entries, parity.oracle_freqs(wl), 0, parity.FactCache(wl))


def test_batched_mode_needs_fp16_embeddings():
    gh.ensure_built()
    from kv_cache_injection_gb300 import _lib, api
    wl = workloads.get("tiny")                      # fp32 embeddings
    store = staging.load_store(wl, api)
    try:
        with pytest.raises(api.ISError) as e:
            api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_BATCHED)
        assert e.value.status == 8
    finally:
        store.destroy()
