"""Store offloaded to host DRAM (kv_placement = IS_KV_HOST): the arena is
page-locked host memory read by the injection kernel over the CPU-GPU link.

InferScale ("Résultats", Scalabilité) offloads the KV store to host memory to go past
the GPU's capacity.  The arithmetic is the device path's, so besides the
oracle checks the injected cache must equal, byte for byte, what the same
calls write from a device-resident store.
"""
import numpy as np
import pytest

from synth import staging, workloads
from tests import gpu_helpers as gh
from tests import parity

pytestmark = pytest.mark.gpu


def _raw(cache):
    """Raw storage bits, so canary NaNs compare equal to themselves."""
    import torch
    return cache.view(torch.int32 if cache.element_size() == 4 else torch.int16)


@pytest.fixture(scope="module")
def api():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api as a
    return a


def _spec(name, **kw):
    base = dict(num_layers=3, num_kv_heads=2, head_dim=128, kv_dtype="bf16",
                rope=workloads.RopeSpec(theta=1.0e4), n_users=6, facts_per_user=150,
                length_dist=("uniform", 1, 12), emb_dim=128, emb_dtype="f16", n_queries=6, k=24,
                query_kind="planted", start=("uniform", 0, 700), block_size=16, tokens_cap=24 * 12,
                block_layout="free_list", seed=77)
    base.update(kw)
    return workloads.WorkloadSpec(name=name, **base)


# NeoX with partner vectors in other lanes (shuffle) and, at a half head of
# exactly 32 vectors, in the same lane's neighbouring register; interleaved;
# all three element types.
SHAPES = [
    _spec("host_bf16_neox"),
    _spec("host_bf16_neox_d512", head_dim=512, num_kv_heads=1, seed=78),
    _spec("host_f32_neox_d256", head_dim=256, num_kv_heads=1, kv_dtype="f32", emb_dtype="f32", seed=79),
    _spec("host_f16_interleaved", kv_dtype="f16", rope=workloads.RopeSpec(theta=5.0e5, style=1), seed=80),
    _spec("host_bf16_llama_scaling", num_kv_heads=4, rope=workloads.LLAMA31_ROPE, seed=81),
]


@pytest.mark.parametrize("spec", SHAPES, ids=[s.name for s in SHAPES])
def test_host_store_matches_oracle_and_device_store(api, spec):
    import torch
    wl = workloads.generate(spec)
    host = staging.load_store(wl, api, kv_placement="host")
    dev = staging.load_store(wl, api)
    try:
        assert api.is_store_info(host)["kv_placement"] == 1
        assert api.is_store_info(dev)["kv_placement"] == 0
        st = gh.check_fused_workload(api, wl, host, sample_tokens=200)
        assert st["tokens"] > 0
        inp = staging.device_inputs(wl)
        ref = staging.canary_cache(wl)
        out = gh.run_fused(api, dev, wl, inp, ref)
        assert out["status"] == 0
        assert torch.equal(_raw(st["cache"]), _raw(ref))
    finally:
        host.destroy()
        dev.destroy()


def test_host_store_llama31_8b(api):
    """The Llama-3.1-8B KV shape (32 layers, 8 KV heads, k = 50) from host memory."""
    wl = workloads.get("llama31_8b")
    host = staging.load_store(wl, api, kv_placement="host")
    try:
        st = gh.check_fused_workload(api, wl, host, all_tokens=True)
        assert st["tokens"] > 50 * 10
        assert st["n"] == st["tokens"] * wl.spec.token_elems      # every injected key element
    finally:
        host.destroy()


def test_host_store_layerwise(api):
    """is_inject_layer from a host store: each layer into its own cache tensor
    equals the corresponding layer of the whole-cache injection."""
    import torch
    wl = workloads.generate(SHAPES[0])
    host = staging.load_store(wl, api, kv_placement="host")
    try:
        st = gh.check_fused_workload(api, wl, host)
        full = st["cache"]
        inp = staging.device_inputs(wl)
        rope = staging.rope_params(wl, api)
        cdesc = api.make_cache_desc(wl.spec.block_size, full.shape[2], wl.spec.kv_dtype)
        Q, k = wl.spec.n_queries, wl.spec.k
        ids = torch.empty((Q, k), dtype=torch.int64, device="cuda")
        sc = torch.empty((Q, k), dtype=torch.float32, device="cuda")
        api.is_retrieve_topk(host, inp["users"], inp["q_emb"], k, ids, sc)
        n_ids = torch.full((Q,), k, dtype=torch.int32, device="cuda")
        for layer in range(wl.spec.num_layers):
            lc = staging.canary_cache(wl)[0].contiguous()       # [2][NB][bs][H][D]
            api.is_inject_layer(host, layer, Q, inp["seg_start"], rope, inp["block_table"], cdesc, lc,
                                fact_ids=ids, n_ids=n_ids, users=inp["users"])
            assert api.is_get_status(host) == 0
            assert torch.equal(_raw(lc), _raw(full[layer]))
    finally:
        host.destroy()


def test_host_store_rejects_bad_placement(api):
    wl = workloads.get("tiny")
    with pytest.raises(api.ISError) as e:
        staging.load_store(wl, api, kv_placement=2)
    assert e.value.status == 1


@pytest.mark.parametrize("cache_dtype,scales", [(None, (1.0, 1.0)), ("e4m3", (0.37, 1.9))], ids=["bf16", "e4m3"])
def test_host_buffer_call_on_host_store(api, cache_dtype, scales):
    """is_retrieve_and_inject_host on a store in host DRAM (the host-memory
    inject kernel, which also writes the call's completion word): the ids,
    scores, segment lengths and every cache byte equal the device call on a
    device-resident store, call after call."""
    import torch
    wl = workloads.generate(SHAPES[0])
    s = wl.spec
    host = staging.load_store(wl, api, kv_placement="host")
    dev = staging.load_store(wl, api)
    try:
        inp = staging.device_inputs(wl)
        ref = staging.canary_cache(wl, cache_dtype=cache_dtype)
        out = gh.run_fused(api, dev, wl, inp, ref, cache_dtype=cache_dtype, k_scale=scales[0], v_scale=scales[1])
        assert out["status"] == 0
        rope = staging.rope_params(wl, api)
        cd = api.make_cache_desc(s.block_size, wl.num_blocks, cache_dtype or s.kv_dtype, scales[0], scales[1])
        Q, k = s.n_queries, s.k
        users = np.array(wl.users, dtype=np.int32)
        q = np.array(wl.queries, dtype=np.float16)
        start = np.array(wl.seg_start, dtype=np.int32)
        bt = np.array(wl.block_table, dtype=np.int32)
        for _ in range(2):
            cache = staging.canary_cache(wl, cache_dtype=cache_dtype)
            ids = np.full((Q, k), -5, dtype=np.int64)
            sc = np.zeros((Q, k), dtype=np.float32)
            ln = np.full(Q, -5, dtype=np.int32)
            api.is_retrieve_and_inject_host(host, users, q, k, start, rope, bt, cd, cache, ids, sc, ln)
            assert np.array_equal(ids, out["ids"])
            assert np.array_equal(sc.view(np.uint32), out["scores"].view(np.uint32))
            assert np.array_equal(ln, out["seg_len"])
            if cache_dtype:
                assert torch.equal(cache, ref)
            else:
                assert torch.equal(_raw(cache), _raw(ref))
        assert api.is_get_status(host) == 0
    finally:
        host.destroy()
        dev.destroy()
