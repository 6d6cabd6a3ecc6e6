"""Query and embedding normalisation (cosine retrieval) on inputs that are not unit length.

Retrieval ranks a user's facts by the cosine of the query with each stored
embedding (InferScale abstract: an embedding is stored with each fact;
"Conception de Système Native au GPU": GPU-resident semantic retrieval).  The
cosine divides by both norms, so neither the query nor the stored rows need to
be unit vectors, and a zero vector scores 0.  Every other workload feeds unit
rows, where a kernel that skipped either division would still pass: here each
stored embedding and each query is scaled by its own factor drawn log-uniformly
from [1e-2, 1e2], one stored row per user is all zeros (the planted fact of a
query, so it would rank first if its norm were ignored) and one query is all
zeros.  Both retrieval paths (per-query GEMV and tensor-core batched) and the
fused retrieve + inject are compared with the oracle element by element.

``test_scaled_inputs_expose_a_missing_norm`` (CPU) checks on the same inputs
that an oracle with either norm dropped disagrees with the true cosine by far
more than the score tolerance, so these inputs do test the normalisation.
"""
import numpy as np
import pytest

from oracle import retrieval
from synth import staging, workloads
from tests import gpu_helpers as gh
from tests import parity


def _spec(facts_per_user: int) -> workloads.WorkloadSpec:
    return workloads.WorkloadSpec(
        name=f"norms_{facts_per_user}", num_layers=2, num_kv_heads=4, head_dim=64, kv_dtype="bf16",
        rope=workloads.RopeSpec(theta=1.0e4), n_users=2, facts_per_user=facts_per_user,
        length_dist=("uniform", 1, 6), emb_dim=256, emb_dtype="f16", n_queries=40, k=16,
        query_kind="planted", start=("uniform", 0, 200), block_size=16, tokens_cap=64 * 6,
        block_layout="free_list", queries_share_user=True, seed=70 + facts_per_user % 7)


ZERO_QUERY = 3


def scaled_workload(facts_per_user: int):
    """The workload with every embedding row and query scaled by 10^U(-2, 2),
    one zero row per user and one zero query.  Queries alternate between the
    two users; even queries are planted on user 0's facts."""
    wl = workloads.generate(_spec(facts_per_user))
    rng = np.random.default_rng(1000 + facts_per_user)
    n, Q = wl.spec.n_facts, wl.spec.n_queries
    wl.users[:] = np.arange(Q, dtype=np.int32) % 2
    fe = 10.0 ** rng.uniform(-2.0, 2.0, size=n)
    wl.emb = (wl.emb.astype(np.float64) * fe[:, None]).astype(np.float16)
    # zero rows: the planted fact of query 0 (user 0) and one fact of user 1
    zero_rows = [int(wl.planted[0]), wl.spec.facts_per_user + 5]
    wl.emb[zero_rows] = 0
    fq = 10.0 ** rng.uniform(-2.0, 2.0, size=Q)
    wl.queries = (wl.queries.astype(np.float64) * fq[:, None]).astype(np.float16)
    wl.queries[ZERO_QUERY] = 0
    wl.extra["zero_rows"] = zero_rows
    return wl


def test_scaled_inputs_expose_a_missing_norm():
    """On the scaled inputs, cosines computed without 1/|e| or without 1/|q|
    differ from the true cosines by far more than the 1e-5 score tolerance for
    almost every row, and change the top-k of almost every query."""
    wl = scaled_workload(700)
    moved = 0
    for q in range(wl.spec.n_queries):
        if q == ZERO_QUERY:
            continue
        facts = wl.user_facts(int(wl.users[q]))
        x = wl.emb[facts].astype(np.float64)
        qq = wl.queries[q].astype(np.float64)
        true = retrieval.cosine_scores(qq, x)
        nx = np.linalg.norm(x, axis=1)
        no_e = (x @ qq) / np.linalg.norm(qq)
        no_q = np.where(nx > 0, (x @ qq) / np.where(nx > 0, nx, 1), 0.0)
        assert np.mean(np.abs(no_e - true) > 1e-3) > 0.9
        assert abs(np.linalg.norm(qq) - 1.0) < 0.5 or np.mean(np.abs(no_q - true) > 1e-3) > 0.9
        ids_true = set(retrieval.topk(true, facts, 16)[0].tolist())
        moved += ids_true != set(retrieval.topk(no_e, facts, 16)[0].tolist())
    assert moved >= wl.spec.n_queries - 2
    # the zero row would otherwise be its planted query's best match
    q0 = wl.queries[0].astype(np.float64)
    assert wl.extra["zero_rows"][0] in wl.user_facts(0)
    assert retrieval.cosine_scores(q0, np.zeros((1, wl.spec.emb_dim)))[0] == 0.0


def _mode(api, store, mode):
    from kv_cache_injection_gb300 import _lib
    api.is_set_retrieval_mode(store, {"auto": _lib.IS_RETRIEVAL_AUTO,
                                      "per_query": _lib.IS_RETRIEVAL_PER_QUERY,
                                      "batched": _lib.IS_RETRIEVAL_BATCHED}[mode])


@pytest.fixture(scope="module", params=[700, 2500])
def env(request):
    gh.ensure_built()
    from kv_cache_injection_gb300 import api
    wl = scaled_workload(request.param)
    store = staging.load_store(wl, api, max_k=1024)
    yield api, wl, store
    store.destroy()


def _retrieve(api, store, wl, k):
    import torch
    inp = staging.device_inputs(wl)
    Q = wl.spec.n_queries
    ids = torch.full((Q, k), -7, dtype=torch.int64, device="cuda")
    sc = torch.zeros((Q, k), dtype=torch.float32, device="cuda")
    api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
    bits = api.is_get_status(store)
    return ids.cpu().numpy(), sc.cpu().numpy(), bits


def _check_retrieval(wl, ids, sc, k):
    for q in range(wl.spec.n_queries):
        o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, k)
        parity.check_topk(ids[q], sc[q], o_ids, o_sc, score_of, k)
        facts = wl.user_facts(int(wl.users[q]))
        n = min(k, len(facts))
        if q == ZERO_QUERY:
            # every cosine is 0: the k lowest ids, in ascending order, exactly 0
            assert np.array_equal(ids[q][:n], facts[:n])
            assert np.all(sc[q][:n] == 0.0)
    for f in wl.extra["zero_rows"]:
        hit = np.argwhere(ids == f)
        for q, r in hit:
            assert sc[q, r] == 0.0, (f, q, sc[q, r])


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["per_query", "batched"])
@pytest.mark.parametrize("k", [16, 1024])
def test_retrieve_topk_unnormalised(env, mode, k):
    api, wl, store = env
    _mode(api, store, mode)
    try:
        ids, sc, bits = _retrieve(api, store, wl, k)
    finally:
        _mode(api, store, "auto")
    assert bits == 0, hex(bits)
    _check_retrieval(wl, ids, sc, k)
    if k >= wl.spec.facts_per_user:
        # the whole ranking came back: each zero row is there, scored exactly 0
        for f in wl.extra["zero_rows"]:
            assert (ids == f).sum() == wl.spec.n_queries // 2


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["per_query", "batched"])
def test_fused_unnormalised(env, mode):
    api, wl, store = env
    _mode(api, store, mode)
    try:
        res = gh.check_fused_workload(api, wl, store, all_tokens=True)
    finally:
        _mode(api, store, "auto")
    assert res["n"] == res["tokens"] * wl.spec.token_elems
