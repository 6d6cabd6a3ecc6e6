"""Device-detected errors: the bad write is skipped, a status bit is latched,
the rest of the call completes and no other cache row changes.  Errors are
made on the host side (bad ids, short block tables, bad users); nothing here
faults, traps or hangs the GPU."""
import numpy as np
import pytest

from synth import staging, workloads
from tests import gpu_helpers as gh
from tests import parity

pytestmark = pytest.mark.gpu

SPEC = workloads.WorkloadSpec(
    name="err_bf16", num_layers=2, num_kv_heads=4, head_dim=64, kv_dtype="bf16",
    rope=workloads.RopeSpec(theta=1.0e4), n_users=2, facts_per_user=40,
    length_dist=("uniform", 3, 9), emb_dim=64, emb_dtype="f16", n_queries=2, k=4,
    query_kind="planted", start=("const", 5), block_size=16, tokens_cap=4 * 9,
    block_layout="free_list", seed=21)


@pytest.fixture(scope="module")
def env():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api
    wl = workloads.generate(SPEC)
    store = staging.load_store(wl, api)
    yield api, wl, store
    store.destroy()


def _inject(api, wl, store, ids, n_ids, users=None, seg_start=None, block_table=None,
            num_blocks=None):
    import torch
    inp = staging.device_inputs(wl)
    cache = staging.canary_cache(wl, num_blocks=num_blocks)
    R = ids.shape[0]
    seg_len = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    slots = torch.full((R * ids.shape[1] * 9 + 1,), -9, dtype=torch.int64, device="cuda")
    api.is_inject(store, torch.from_numpy(ids).cuda(), torch.from_numpy(n_ids).cuda(),
                  inp["seg_start"] if seg_start is None else torch.from_numpy(seg_start).cuda(),
                  staging.rope_params(wl, api),
                  inp["block_table"] if block_table is None else torch.from_numpy(block_table).cuda(),
                  api.make_cache_desc(16, cache.shape[2], "bf16"), cache,
                  users=None if users is None else torch.from_numpy(users).cuda(),
                  seg_len_out=seg_len, slot_mapping_out=slots)
    bits = api.is_get_status(store)
    return bits, cache, seg_len.cpu().numpy(), slots.cpu().numpy()


def _valid_compare(wl, cache, rows, seg_len, slots):
    plans, lens = parity.oracle_plans(wl, rows)
    assert np.array_equal(seg_len, lens)
    want = np.concatenate([[e[3] for e in pl] for pl in plans]).astype(np.int64)
    assert np.array_equal(slots[: len(want)], want)
    entries = [e for pl in plans for e in pl]
    gk, gv = gh.gather_rows(cache, [e[3] for e in entries])
    parity.compare_tokens(wl, gk, gv, entries, parity.oracle_freqs(wl), 0, parity.FactCache(wl))
    gh.assert_only_slots_changed(cache, "bf16", want)


def test_out_of_range_fact_contributes_nothing(env):
    from kv_cache_injection_gb300 import _lib
    api, wl, store = env
    ids = np.array([[3, 999, 7, -2], [41, 42, 43, 44]], dtype=np.int64)
    n_ids = np.array([4, 4], dtype=np.int32)
    bits, cache, seg_len, slots = _inject(api, wl, store, ids, n_ids)
    assert bits == _lib.IS_ST_FACT_RANGE
    _valid_compare(wl, cache, [[3, 7], [41, 42, 43, 44]], seg_len, slots)


def test_fact_of_another_user(env):
    from kv_cache_injection_gb300 import _lib
    api, wl, store = env
    ids = np.array([[3, 45, 7, 8], [41, 42, 2, 44]], dtype=np.int64)
    bits, cache, seg_len, slots = _inject(api, wl, store, ids, np.array([4, 4], np.int32),
                                          users=np.array([0, 1], np.int32))
    assert bits == _lib.IS_ST_FACT_USER
    _valid_compare(wl, cache, [[3, 7, 8], [41, 42, 44]], seg_len, slots)


def test_block_table_too_short_and_bad_block(env):
    from kv_cache_injection_gb300 import _lib
    api, wl, store = env
    ids = np.array([[1, 2, 3, 4], [41, 42, 43, 44]], dtype=np.int64)
    bt = wl.block_table.copy()
    # request 0: only logical block 0 is mapped (a 1-wide table), request 1: a bad block id
    bt1 = bt[:, :1].copy()
    bits, cache, seg_len, slots = _inject(api, wl, store, ids, np.array([4, 4], np.int32),
                                          block_table=np.ascontiguousarray(bt1))
    assert bits & _lib.IS_ST_BLOCK_TABLE
    seg0 = int(seg_len[0])
    # positions 5..15 (block 0) were written, the rest skipped with slot -1
    assert np.all(slots[: 16 - 5] >= 0) and np.all(slots[16 - 5: seg0] == -1)
    bt2 = bt.copy()
    bt2[1, 1] = wl.num_blocks + 5
    bits, cache, seg_len, slots = _inject(api, wl, store, ids, np.array([4, 4], np.int32),
                                          block_table=bt2)
    assert bits == _lib.IS_ST_BLOCK_ID
    s1 = slots[int(seg_len[0]): int(seg_len.sum())]
    assert np.all(s1[16 - 5: 32 - 5] == -1) and np.all(s1[: 16 - 5] >= 0)


def test_bad_counts_and_positions(env):
    from kv_cache_injection_gb300 import _lib
    api, wl, store = env
    ids = np.array([[1, 2, 3, 4], [41, 42, 43, 44]], dtype=np.int64)
    bits, cache, seg_len, _ = _inject(api, wl, store, ids, np.array([5, 2], np.int32))
    assert bits == _lib.IS_ST_COUNT and seg_len[0] == 0 and seg_len[1] > 0
    bits, cache, seg_len, _ = _inject(api, wl, store, ids, np.array([4, 4], np.int32),
                                      seg_start=np.array([-3, 5], np.int32))
    assert bits == _lib.IS_ST_POSITION and seg_len[0] == 0 and seg_len[1] > 0


def test_bad_user_in_retrieval(env):
    import torch
    from kv_cache_injection_gb300 import _lib
    api, wl, store = env
    inp = staging.device_inputs(wl)
    users = torch.tensor([0, 7], dtype=torch.int32, device="cuda")
    ids = torch.empty((2, 4), dtype=torch.int64, device="cuda")
    sc = torch.empty((2, 4), dtype=torch.float32, device="cuda")
    api.is_retrieve_topk(store, users, inp["q_emb"], 4, ids, sc)
    assert api.is_get_status(store) == _lib.IS_ST_USER_RANGE
    g = ids.cpu().numpy()
    assert np.all(g[1] == -1) and np.all(g[0] >= 0)


def test_host_validation_errors(env):
    import torch
    api, wl, store = env
    inp = staging.device_inputs(wl)
    ids = torch.empty((2, 4), dtype=torch.int64, device="cuda")
    sc = torch.empty((2, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(api.ISError) as e:
        api.is_retrieve_topk(store, inp["users"], inp["q_emb"], 5, ids, sc)   # k > max_k
    assert e.value.status == 4
    cache = staging.canary_cache(wl)
    bad = api.make_cache_desc(16, cache.shape[2], "f32")                      # dtype mismatch
    with pytest.raises(api.ISError) as e:
        api.is_retrieve_and_inject(store, inp["users"], inp["q_emb"], 4, inp["seg_start"],
                                   staging.rope_params(wl, api), inp["block_table"], bad, cache)
    assert e.value.status == 1
    with pytest.raises(api.ISError) as e:                                      # capacity
        k = torch.zeros((1, 2, 4, 64), dtype=torch.bfloat16, device="cuda")
        api.is_store_add_facts(store, 0, [1], k, k, torch.zeros((1, 64), dtype=torch.float16,
                                                                 device="cuda"))
    assert e.value.status == 3
    assert api.is_get_status(store) == 0


def test_bad_user_in_one_user_store():
    """A store of one user, queried with users out of range next to valid
    ones: each bad row gets the status bit and the empty result, and every
    other row, call after call, still matches the oracle (the cosine bins
    are left clean between calls)."""
    import torch
    from kv_cache_injection_gb300 import _lib
    from kv_cache_injection_gb300 import api
    gh.ensure_built()
    wl = workloads.get("tiny")
    store = staging.load_store(wl, api, max_queries=4)
    try:
        q = torch.from_numpy(np.repeat(wl.queries, 3, axis=0)).cuda()
        k = wl.spec.k
        for users, bad in (([0, 3, 0], {1}), ([-1, 0, 1], {0, 2}), ([0, 0, 0], set())):
            u = torch.tensor(users, dtype=torch.int32, device="cuda")
            ids = torch.full((3, k), -7, dtype=torch.int64, device="cuda")
            sc = torch.zeros((3, k), dtype=torch.float32, device="cuda")
            api.is_retrieve_topk(store, u, q, k, ids, sc)
            bits = api.is_get_status(store)
            assert bits == (_lib.IS_ST_USER_RANGE if bad else 0), hex(bits)
            g, s = ids.cpu().numpy(), sc.cpu().numpy()
            o_ids, o_sc, score_of = parity.oracle_retrieve(wl, 0, k)
            for r in range(3):
                if r in bad:
                    assert np.all(g[r] == -1) and np.all(np.isneginf(s[r]))
                else:
                    parity.check_topk(g[r], s[r], o_ids, o_sc, score_of, k)
    finally:
        store.destroy()
