"""Injection into an FP8 E4M3 paged cache (vLLM's 8-bit KV cache) from a
bf16 / fp16 store: each rotated key element and value element is stored as
E4M3(x * fp32(1 / scale)), rounded to nearest even and saturated to +-448.

V bytes are compared bit for bit with the oracle (which takes the same fp32
product); keys within one E4M3 ulp of the oracle's fp64 rotation.
"""
import numpy as np
import pytest

from synth import staging, workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


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
                block_layout="free_list", seed=90)
    base.update(kw)
    return workloads.WorkloadSpec(name=name, **base)


SHAPES = [
    _spec("fp8_bf16_neox"),
    _spec("fp8_f16_interleaved", kv_dtype="f16", rope=workloads.RopeSpec(theta=5.0e5, style=1), seed=91),
    _spec("fp8_bf16_llama_scaling_d256", head_dim=256, num_kv_heads=1, rope=workloads.LLAMA31_ROPE, seed=92),
]
# (k_scale, v_scale): vLLM's default, non-power-of-two scales, and a V scale
# small enough that N(0, 1) values saturate.
SCALES = [(1.0, 1.0), (0.37, 1.9), (0.8, 0.004)]


@pytest.mark.parametrize("placement", ["device", "host"])
@pytest.mark.parametrize("scales", SCALES, ids=["unit", "odd", "saturating"])
@pytest.mark.parametrize("spec", SHAPES, ids=[s.name for s in SHAPES])
def test_fp8_cache_matches_oracle(api, spec, scales, placement):
    wl = workloads.generate(spec)
    store = staging.load_store(wl, api, kv_placement=placement)
    try:
        st = gh.check_fused_workload(api, wl, store, sample_tokens=120, cache_dtype="e4m3",
                                     k_scale=scales[0], v_scale=scales[1])
        assert st["tokens"] > 0 and st["n"] > 0
        if scales[1] < 0.01:
            assert st["v_saturated"] > 0
    finally:
        store.destroy()


def test_fp8_cache_llama31_8b(api):
    """The Llama-3.1-8B KV shape at k = 50 into an FP8 cache."""
    wl = workloads.get("llama31_8b")
    store = staging.load_store(wl, api)
    try:
        st = gh.check_fused_workload(api, wl, store, cache_dtype="e4m3", k_scale=0.5, v_scale=0.75,
                                     all_tokens=True)
        assert st["tokens"] > 50 * 10
        assert st["n"] == st["tokens"] * wl.spec.token_elems      # every injected key element
    finally:
        store.destroy()


def test_fp8_layerwise_equals_whole(api):
    """is_inject_layer into per-layer FP8 caches equals the whole-cache injection."""
    import torch
    wl = workloads.generate(SHAPES[0])
    store = staging.load_store(wl, api)
    try:
        st = gh.check_fused_workload(api, wl, store, cache_dtype="e4m3", k_scale=0.37, v_scale=1.9)
        full = st["cache"]
        inp = staging.device_inputs(wl)
        rope = staging.rope_params(wl, api)
        cd = api.make_cache_desc(wl.spec.block_size, full.shape[2], "e4m3", 0.37, 1.9)
        Q, k = wl.spec.n_queries, wl.spec.k
        ids = torch.empty((Q, k), dtype=torch.int64, device="cuda")
        sc = torch.empty((Q, k), dtype=torch.float32, device="cuda")
        api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
        n_ids = torch.full((Q,), k, dtype=torch.int32, device="cuda")
        for layer in range(wl.spec.num_layers):
            lc = staging.canary_cache(wl, cache_dtype="e4m3")[0].contiguous()
            api.is_inject_layer(store, layer, Q, inp["seg_start"], rope, inp["block_table"], cd, lc,
                                fact_ids=ids, n_ids=n_ids, users=inp["users"])
            assert api.is_get_status(store) == 0
            assert torch.equal(lc, full[layer])
    finally:
        store.destroy()


def test_fp8_cache_rejections(api):
    import torch
    wl = workloads.get("tiny")                       # fp32 store
    store = staging.load_store(wl, api)
    try:
        inp = staging.device_inputs(wl)
        cache = staging.canary_cache(wl, cache_dtype="e4m3")
        rope = staging.rope_params(wl, api)
        ids = torch.zeros((1, wl.spec.k), dtype=torch.int64, device="cuda")
        sc = torch.zeros((1, wl.spec.k), dtype=torch.float32, device="cuda")
        cd = api.make_cache_desc(wl.spec.block_size, cache.shape[2], "e4m3")
        with pytest.raises(api.ISError) as e:
            api.is_retrieve_and_inject(store, inp["users"], inp["q_emb"], wl.spec.k, inp["seg_start"], rope,
                                       inp["block_table"], cd, cache, ids, sc)
        assert e.value.status == 8
    finally:
        store.destroy()
    wl = workloads.generate(SHAPES[0])
    store = staging.load_store(wl, api)
    try:
        inp = staging.device_inputs(wl)
        cache = staging.canary_cache(wl, cache_dtype="e4m3")
        rope = staging.rope_params(wl, api)
        Q, k = wl.spec.n_queries, wl.spec.k
        ids = torch.zeros((Q, k), dtype=torch.int64, device="cuda")
        sc = torch.zeros((Q, k), dtype=torch.float32, device="cuda")
        for ks, vs in [(0.0, 1.0), (1.0, float("inf")), (-1.0, 1.0)]:
            cd = api.make_cache_desc(wl.spec.block_size, cache.shape[2], "e4m3", ks, vs)
            with pytest.raises(api.ISError) as e:
                api.is_retrieve_and_inject(store, inp["users"], inp["q_emb"], k, inp["seg_start"], rope,
                                           inp["block_table"], cd, cache, ids, sc)
            assert e.value.status == 1
        assert np.all(staging.cache_bits(cache) == 0x7F)
    finally:
        store.destroy()
