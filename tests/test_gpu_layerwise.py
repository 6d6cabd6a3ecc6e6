"""Layer-wise injection (is_inject_layer) into per-layer cache tensors, as a
layer-by-layer KV connector would call it: the first call plans the segments,
the others reuse the plan.  Every layer must equal, bit for bit, that layer
of a whole-model injection (which the other tests pin to the oracle)."""
import numpy as np
import pytest

from synth import staging, workloads
from tests import gpu_helpers as gh
from tests import parity

pytestmark = pytest.mark.gpu

SPEC = workloads.WorkloadSpec(
    name="layerwise", num_layers=5, num_kv_heads=4, head_dim=128, kv_dtype="bf16",
    rope=workloads.LLAMA31_ROPE, n_users=2, facts_per_user=300, length_dist=("uniform", 3, 30),
    emb_dim=128, emb_dtype="f16", n_queries=2, k=12, query_kind="planted",
    start=("uniform", 0, 200), block_size=16, tokens_cap=12 * 30, block_layout="free_list", seed=51)


@pytest.fixture(scope="module")
def env():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api
    wl = workloads.generate(SPEC)
    store = staging.load_store(wl, api)
    yield api, wl, store
    store.destroy()


def _layer_caches(wl):
    import torch
    s = wl.spec
    shape = (2, wl.num_blocks, s.block_size, s.num_kv_heads, s.head_dim)
    out = []
    for _ in range(s.num_layers):
        c = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        staging.refill_canary(c, "bf16")
        out.append(c)
    return out


def test_layerwise_equals_whole_injection(env):
    import torch
    api, wl, store = env
    s = wl.spec
    rng = np.random.default_rng(3)
    R, stride = 2, s.k
    n_ids = np.array([12, 7], dtype=np.int32)
    ids = np.full((R, stride), -1, dtype=np.int64)
    for r in range(R):
        ids[r, :n_ids[r]] = rng.choice(wl.user_facts(int(wl.users[r])), size=n_ids[r], replace=False)
    d_ids, d_n = torch.from_numpy(ids).cuda(), torch.from_numpy(n_ids).cuda()
    inp = staging.device_inputs(wl)
    rope = staging.rope_params(wl, api)
    cd = api.make_cache_desc(s.block_size, wl.num_blocks, "bf16")
    whole = staging.canary_cache(wl)
    len_w = torch.empty(R, dtype=torch.int32, device="cuda")
    slots_w = torch.full((R * stride * 30,), -9, dtype=torch.int64, device="cuda")
    api.is_inject(store, d_ids, d_n, inp["seg_start"], rope, inp["block_table"], cd, whole,
                  users=inp["users"], seg_len_out=len_w, slot_mapping_out=slots_w)
    layers = _layer_caches(wl)
    len_l = torch.empty(R, dtype=torch.int32, device="cuda")
    slots_l = torch.full_like(slots_w, -9)
    for l in range(s.num_layers):
        if l == 0:
            api.is_inject_layer(store, 0, R, inp["seg_start"], rope, inp["block_table"], cd, layers[0],
                                fact_ids=d_ids, n_ids=d_n, users=inp["users"], seg_len_out=len_l,
                                slot_mapping_out=slots_l)
        else:
            api.is_inject_layer(store, l, R, inp["seg_start"], rope, inp["block_table"], cd, layers[l])
    assert api.is_get_status(store) == 0
    assert torch.equal(len_w, len_l)
    assert torch.equal(slots_w, slots_l)
    for l in range(s.num_layers):
        assert torch.equal(whole[l].view(torch.int16), layers[l].view(torch.int16)), f"layer {l}"
    # and the whole injection against the oracle
    plans, lens = parity.oracle_plans(wl, [ids[r, :n_ids[r]] for r in range(R)])
    assert np.array_equal(len_w.cpu().numpy(), lens)
    entries = [e for pl in plans for e in pl]
    gk, gv = gh.gather_rows(whole, [e[3] for e in entries])
    parity.compare_tokens(wl, gk, gv, entries, parity.oracle_freqs(wl), 0, parity.FactCache(wl))


def test_retrieve_then_layerwise_equals_fused(env):
    import torch
    api, wl, store = env
    s = wl.spec
    inp = staging.device_inputs(wl)
    k = s.k
    fused = staging.canary_cache(wl)
    out = gh.run_fused(api, store, wl, inp, fused)
    assert out["status"] == 0
    ids = torch.empty((2, k), dtype=torch.int64, device="cuda")
    sc = torch.empty((2, k), dtype=torch.float32, device="cuda")
    api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
    n_ids = (ids >= 0).sum(1).to(torch.int32)
    rope = staging.rope_params(wl, api)
    cd = api.make_cache_desc(s.block_size, wl.num_blocks, "bf16")
    layers = _layer_caches(wl)
    for l in range(s.num_layers):
        api.is_inject_layer(store, l, 2, inp["seg_start"], rope, inp["block_table"], cd, layers[l],
                            fact_ids=ids if l == 0 else None, n_ids=n_ids if l == 0 else None)
    assert api.is_get_status(store) == 0
    for l in range(s.num_layers):
        assert torch.equal(fused[l].view(torch.int16), layers[l].view(torch.int16)), f"layer {l}"


def test_reuse_needs_a_plan_of_the_same_size(env):
    api, wl, store = env
    s = wl.spec
    inp = staging.device_inputs(wl)
    rope = staging.rope_params(wl, api)
    cd = api.make_cache_desc(s.block_size, wl.num_blocks, "bf16")
    layers = _layer_caches(wl)
    with pytest.raises(api.ISError) as e:
        api.is_inject_layer(store, 1, 1, inp["seg_start"][:1], rope, inp["block_table"][:1], cd, layers[1])
    assert e.value.status == 1
    with pytest.raises(api.ISError) as e:
        api.is_inject_layer(store, s.num_layers, 2, inp["seg_start"], rope, inp["block_table"], cd, layers[0])
    assert e.value.status == 4


def test_layer_groups_equal_the_fused_call(env):
    """is_inject_layers: all layers into per-layer tensors in one launch (with
    planning), then groups of layers reusing the plan, each equal byte for byte
    to the fused call's layers.  The per-layer tensors are allocated one by one
    (arbitrary addresses, the way an engine keeps them)."""
    import torch
    api, wl, store = env
    s = wl.spec
    inp = staging.device_inputs(wl)
    k = s.k
    fused = staging.canary_cache(wl)
    out = gh.run_fused(api, store, wl, inp, fused)
    assert out["status"] == 0
    ids = torch.empty((2, k), dtype=torch.int64, device="cuda")
    sc = torch.empty((2, k), dtype=torch.float32, device="cuda")
    api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
    n_ids = (ids >= 0).sum(1).to(torch.int32)
    rope = staging.rope_params(wl, api)
    cd = api.make_cache_desc(s.block_size, wl.num_blocks, "bf16")
    layers = _layer_caches(wl)
    api.is_inject_layers(store, 0, 2, inp["seg_start"], rope, inp["block_table"], cd, layers,
                         fact_ids=ids, n_ids=n_ids)
    assert api.is_get_status(store) == 0
    for l in range(s.num_layers):
        assert torch.equal(fused[l].view(torch.int16), layers[l].view(torch.int16)), f"layer {l}"
    groups = _layer_caches(wl)
    for l0, l1 in ((0, 2), (2, 3), (3, s.num_layers)):
        api.is_inject_layers(store, l0, 2, inp["seg_start"], rope, inp["block_table"], cd, groups[l0:l1])
    assert api.is_get_status(store) == 0
    for l in range(s.num_layers):
        assert torch.equal(fused[l].view(torch.int16), groups[l].view(torch.int16)), f"group layer {l}"
    with pytest.raises(api.ISError):
        api.is_inject_layers(store, 1, 2, inp["seg_start"], rope, inp["block_table"], cd, groups)   # past L
    with pytest.raises(api.ISError):
        api.is_inject_layers(store, 0, 2, inp["seg_start"], rope, inp["block_table"], cd, [])


def test_reuse_after_fused_and_host_calls(env):
    """A layer call may reuse the plan of is_retrieve_and_inject and of
    is_retrieve_and_inject_host, on its mapped path (small inputs) and on its
    copy path (a block table padded past 16 KiB): each reuse puts every layer
    byte for byte where the fused call put it."""
    import torch
    api, wl, store = env
    s = wl.spec
    inp = staging.device_inputs(wl)
    fused = staging.canary_cache(wl)
    out = gh.run_fused(api, store, wl, inp, fused)
    assert out["status"] == 0
    rope = staging.rope_params(wl, api)
    cd = api.make_cache_desc(s.block_size, wl.num_blocks, "bf16")
    Q = len(wl.users)
    users = np.ascontiguousarray(wl.users, dtype=np.int32)
    q = np.ascontiguousarray(wl.queries, dtype=np.float16)
    start = np.ascontiguousarray(wl.seg_start, dtype=np.int32)
    bt0 = np.ascontiguousarray(wl.block_table, dtype=np.int32)
    bt_big = np.ascontiguousarray(np.pad(bt0, ((0, 0), (0, 2048))))
    assert Q * bt_big.shape[1] * 4 > 16384
    for planner in ("fused", "host mapped", "host copy"):
        if planner == "fused":
            gh.run_fused(api, store, wl, inp, staging.canary_cache(wl))
        else:
            bt = bt0 if planner == "host mapped" else bt_big
            ln = np.empty(Q, dtype=np.int32)
            api.is_retrieve_and_inject_host(store, users, q, s.k, start, rope, bt, cd, staging.canary_cache(wl),
                                            seg_len_out=ln)
            assert np.array_equal(ln, out["seg_len"]), planner
        layers = _layer_caches(wl)
        api.is_inject_layers(store, 0, Q, inp["seg_start"], rope, inp["block_table"], cd, layers)
        assert api.is_get_status(store) == 0
        for l in range(s.num_layers):
            assert torch.equal(fused[l].view(torch.int16), layers[l].view(torch.int16)), f"{planner}, layer {l}"
