"""The bounded waits give up without hanging, report IS_ERR_TIMEOUT and leave
the GPU usable.

Every wait inside the store's kernels is bounded.  ``is_set_wait_budget(store,
0)`` makes each wait of the injection pipeline and of the batched
(tensor-core) similarity look once and give up at once if its data has not
landed, which with loads just issued is almost certain; so the time-out path
runs on a healthy GPU, with no fault and no hang.  The kernels must then:
* latch IS_ST_TIMEOUT, so that is_get_status returns IS_ERR_TIMEOUT;
* let the copies and MMAs they already started finish before they exit;
* leave every cache row either as it was (the canary) or holding exactly what
  the oracle says the call writes there;
and the next call with the default budget must be clean and correct.
"""
import numpy as np
import pytest

from synth import staging, workloads
from tests import gpu_helpers as gh
from tests import parity

pytestmark = pytest.mark.gpu

IS_ST_TIMEOUT = 0x80

SPEC = workloads.WorkloadSpec(
    name="timeout", num_layers=4, num_kv_heads=8, head_dim=128, kv_dtype="bf16",
    rope=workloads.RopeSpec(theta=1.0e6), n_users=1, facts_per_user=1500,
    length_dist=("uniform", 10, 40), emb_dim=256, emb_dtype="f16", n_queries=40, k=20,
    query_kind="planted", start=("uniform", 0, 100), block_size=16, tokens_cap=20 * 40,
    block_layout="free_list", queries_share_user=True, seed=91)


@pytest.fixture(scope="module")
def env():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api
    wl = workloads.generate(SPEC)
    store = staging.load_store(wl, api)
    yield api, wl, store
    api.is_set_wait_budget(store, 2_000_000_000)
    store.destroy()


def _status_and_code(api, store):
    """is_get_status through the C ABI: (bits, return code)."""
    import ctypes
    from kv_cache_injection_gb300 import _lib
    bits = ctypes.c_uint32()
    code = _lib.load().is_get_status(ctypes.c_void_p(store.handle), None, ctypes.byref(bits))
    return int(bits.value), int(code)


def _mode(api, store, name):
    from kv_cache_injection_gb300 import _lib
    api.is_set_retrieval_mode(store, {"per_query": _lib.IS_RETRIEVAL_PER_QUERY,
                                      "batched": _lib.IS_RETRIEVAL_BATCHED,
                                      "auto": _lib.IS_RETRIEVAL_AUTO}[name])


def test_budget_range(env):
    from kv_cache_injection_gb300 import api as a
    api, _, store = env
    for bad in (-1, 2_000_000_001):
        with pytest.raises(a.ISError) as e:
            api.is_set_wait_budget(store, bad)
        assert e.value.status == 1


def test_inject_timeout_leaves_canaries_or_correct_rows(env):
    """Per-query retrieval (no waits) then the injection with a zero budget."""
    api, wl, store = env
    _mode(api, store, "per_query")
    inp = staging.device_inputs(wl)
    timed_out = False
    try:
        for attempt in range(3):
            cache = staging.canary_cache(wl)
            api.is_set_wait_budget(store, 0)
            out = gh.run_fused(api, store, wl, inp, cache)
            bits = out["status"]
            assert bits & ~IS_ST_TIMEOUT == 0, hex(bits)
            # the retrieval has no waits: its ids are the oracle's, so the plan is known
            for q in range(wl.spec.n_queries):
                o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, wl.spec.k)
                parity.check_topk(out["ids"][q], out["scores"][q], o_ids, o_sc, score_of, wl.spec.k)
            plans, lens = parity.oracle_plans(wl, out["ids"])
            assert np.array_equal(out["seg_len"], lens)
            entries = [e for pl in plans for e in pl]
            target = np.array([e[3] for e in entries], dtype=np.int64)
            changed = gh.changed_slots(cache, "bf16")                # [L][2][slots]; no partial rows
            outside = changed.copy()
            outside[:, :, target] = False
            assert not outside.any(), "a row outside the segment changed"
            # rows written are the oracle's; K and V of one (token, layer) go together
            written = changed[:, :, target]                          # [L][2][n]
            assert np.array_equal(written[:, 0], written[:, 1])
            idx = np.nonzero(written[:, 0].any(axis=0))[0]
            if len(idx):
                sub = [entries[i] for i in idx]
                gk, gv = gh.gather_rows(cache, [e[3] for e in sub])
                for li in range(wl.spec.num_layers):
                    rows = np.nonzero(written[li, 0, idx])[0]
                    if len(rows) == 0:
                        continue
                    ent = [sub[i] for i in rows]
                    st = parity.compare_runs(wl, gk[rows][:, li:li + 1], gv[rows][:, li:li + 1], ent,
                                             parity.oracle_freqs(wl), wl.spec.rope.style,
                                             _LayerFacts(wl, li))
                    assert st["n"] == len(rows) * wl.spec.num_kv_heads * wl.spec.head_dim
            if bits & IS_ST_TIMEOUT:
                timed_out = True
                break
        assert timed_out, "no wait gave up in three zero-budget calls"
        # the same call with the default budget: clean and complete
        api.is_set_wait_budget(store, 2_000_000_000)
        st = gh.check_fused_workload(api, wl, store, all_tokens=True)
        assert st["n"] == st["tokens"] * wl.spec.token_elems
    finally:
        api.is_set_wait_budget(store, 2_000_000_000)
        _mode(api, store, "auto")


class _LayerFacts:
    """One layer of each fact's K and V ([len][1][H][D]), for comparing the
    rows of that layer alone."""

    def __init__(self, wl, layer):
        self.facts = gh.DeviceFactCache(wl)
        self.layer = layer

    def __call__(self, f):
        K, V = self.facts(f)
        return K[:, self.layer:self.layer + 1], V[:, self.layer:self.layer + 1]


def test_is_get_status_reports_timeout(env):
    """IS_ERR_TIMEOUT and IS_ST_TIMEOUT through the C call itself."""
    import torch
    api, wl, store = env
    _mode(api, store, "per_query")
    inp = staging.device_inputs(wl)
    try:
        for attempt in range(3):
            cache = staging.canary_cache(wl)
            api.is_set_wait_budget(store, 0)
            k = wl.spec.k
            ids = torch.empty((wl.spec.n_queries, k), dtype=torch.int64, device="cuda")
            sc = torch.empty((wl.spec.n_queries, k), dtype=torch.float32, device="cuda")
            sl = torch.empty((wl.spec.n_queries,), dtype=torch.int32, device="cuda")
            api.is_retrieve_and_inject(store, inp["users"], inp["q_emb"], k, inp["seg_start"],
                                       staging.rope_params(wl, api), inp["block_table"],
                                       api.make_cache_desc(wl.spec.block_size, wl.num_blocks, "bf16"),
                                       cache, ids, sc, sl)
            bits, code = _status_and_code(api, store)
            if bits:
                assert bits == IS_ST_TIMEOUT and code == 6                 # IS_ERR_TIMEOUT
                break
            assert code == 0
        else:
            pytest.fail("no wait gave up in three zero-budget calls")
        bits, code = _status_and_code(api, store)                          # cleared by the read
        assert bits == 0 and code == 0
    finally:
        api.is_set_wait_budget(store, 2_000_000_000)
        _mode(api, store, "auto")


def test_batched_similarity_timeout_then_recovers(env):
    """The tensor-core similarity with a zero budget: its CTAs give up, drain
    their TMA loads and MMAs, free their TMEM and exit; the next call with
    the default budget is correct (it also needs that TMEM back)."""
    import torch
    api, wl, store = env
    inp = staging.device_inputs(wl)
    Q, k = wl.spec.n_queries, wl.spec.k

    def retrieve():
        ids = torch.full((Q, k), -7, dtype=torch.int64, device="cuda")
        sc = torch.zeros((Q, k), dtype=torch.float32, device="cuda")
        api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
        return ids, sc

    def check(ids, sc):
        ids, sc = ids.cpu().numpy(), sc.cpu().numpy()
        for q in range(Q):
            o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, k)
            parity.check_topk(ids[q], sc[q], o_ids, o_sc, score_of, k)

    _mode(api, store, "batched")
    try:
        ids, sc = retrieve()                                               # fills the score scratch
        assert _status_and_code(api, store) == (0, 0)
        check(ids, sc)
        for attempt in range(3):
            api.is_set_wait_budget(store, 0)
            retrieve()
            bits, code = _status_and_code(api, store)
            if bits:
                assert bits == IS_ST_TIMEOUT and code == 6
                break
        else:
            pytest.fail("no wait gave up in three zero-budget calls")
        api.is_set_wait_budget(store, 2_000_000_000)
        for _ in range(2):
            ids, sc = retrieve()
            assert _status_and_code(api, store) == (0, 0)
            check(ids, sc)
    finally:
        api.is_set_wait_budget(store, 2_000_000_000)
        _mode(api, store, "auto")
