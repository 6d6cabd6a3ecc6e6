"""The allocation-free entry point, is_inject_noalloc.

Some callers cannot allocate device memory: a serving engine that reserves
all of HBM for its own pools at start-up and hands kernels only memory it
owns, or code running where cudaMalloc is not allowed.  is_inject_noalloc
serves them: the caller keeps the facts' pre-RoPE K and raw V in its own
token-major buffer and passes inputs and outputs; the library creates no store
and keeps the per-request segment plan in a fixed static device array.

This test calls it through the C ABI twice in a row (two different request
batches on the same stream, so the second call overwrites the static array
the first used) and checks each output against the existing is_inject entry
point on a store holding the same facts: values bit for bit, rotated keys
within one bf16 ulp, segment lengths and slot mappings exactly.  It lives in
a file of its own that pytest collects last.
"""
import numpy as np
import pytest

from synth import kvgen, staging, workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

SPEC = workloads.WorkloadSpec(
    name="noalloc_bf16", num_layers=3, num_kv_heads=4, head_dim=64, kv_dtype="bf16",
    rope=workloads.RopeSpec(theta=5e5, scaling=1, factor=8.0, low_freq_factor=1.0,
                            high_freq_factor=4.0, original_max_pos=64),
    n_users=1, facts_per_user=300, length_dist=("uniform", 1, 21), emb_dim=64, emb_dtype="f16",
    n_queries=6, k=12, query_kind="planted", start=("uniform", 0, 500), block_size=16,
    tokens_cap=12 * 21, block_layout="free_list", queries_share_user=True, seed=31)


def _requests(wl, seed):
    rng = np.random.default_rng(seed)
    R, stride = wl.spec.n_queries, wl.spec.k
    n_ids = rng.integers(0, stride + 1, size=R).astype(np.int32)
    ids = np.full((R, stride), -1, dtype=np.int64)
    for r in range(R):
        ids[r, :n_ids[r]] = rng.choice(wl.spec.n_facts, size=n_ids[r], replace=False)
    return ids, n_ids


def test_noalloc_matches_is_inject_on_two_calls_in_a_row():
    import torch
    from kv_cache_injection_gb300 import api
    from oracle import numerics
    gh.ensure_built()
    wl = workloads.generate(SPEC)
    s = wl.spec
    store = staging.load_store(wl, api)
    try:
        # Caller-owned token-major arena [T][L][2][H][D] with the same facts.
        T = wl.total_tokens
        k = torch.empty((T, s.num_layers, s.num_kv_heads, s.head_dim), dtype=torch.bfloat16,
                        device="cuda")
        v = torch.empty_like(k)
        staging.fill_kv(k, "bf16", s.seed, kvgen.STREAM_K, 0)
        staging.fill_kv(v, "bf16", s.seed, kvgen.STREAM_V, 0)
        arena = torch.stack([k, v], dim=2).contiguous()
        fact_tok = torch.from_numpy(wl.tok_base).cuda()
        fact_len = torch.from_numpy(wl.lengths).cuda()
        inp = staging.device_inputs(wl)
        rope = staging.rope_params(wl, api)
        cdesc = api.make_cache_desc(s.block_size, wl.num_blocks, "bf16")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        batches, outs = [], []
        for seed in (1, 2):                       # two calls in a row, same stream
            ids, n_ids = _requests(wl, seed)
            d_ids, d_n = torch.from_numpy(ids).cuda(), torch.from_numpy(n_ids).cuda()
            cache = staging.canary_cache(wl)
            seg_len = torch.full((s.n_queries,), -1, dtype=torch.int32, device="cuda")
            slots = torch.full((s.n_queries * s.k * 21,), -9, dtype=torch.int64, device="cuda")
            api.is_inject_noalloc(arena, fact_tok, fact_len, int(wl.lengths.max()), s.num_layers,
                                  s.num_kv_heads, s.head_dim, "bf16", d_ids, d_n, inp["seg_start"],
                                  rope, inp["block_table"], cdesc, cache, status,
                                  seg_len_out=seg_len, slot_mapping_out=slots)
            batches.append((d_ids, d_n))
            outs.append((cache, seg_len, slots))
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for (d_ids, d_n), (cache, seg_len, slots) in zip(batches, outs):
            ref = staging.canary_cache(wl)
            ref_len = torch.full_like(seg_len, -1)
            ref_slots = torch.full_like(slots, -9)
            api.is_inject(store, d_ids, d_n, inp["seg_start"], rope, inp["block_table"], cdesc, ref,
                          seg_len_out=ref_len, slot_mapping_out=ref_slots)
            assert api.is_get_status(store) == 0
            assert torch.equal(seg_len, ref_len) and int(seg_len.sum()) > 0
            assert torch.equal(slots, ref_slots)
            a = staging.cache_bits(cache)
            b = staging.cache_bits(ref)
            assert np.array_equal(a[:, 1], b[:, 1])                     # V and untouched rows
            ga, gb = numerics.decode(a[:, 0], "bf16"), numerics.decode(b[:, 0], "bf16")
            same = (a[:, 0] == b[:, 0]) | (np.abs(ga - gb) <= numerics.ulp(gb, "bf16"))
            assert same.all()
    finally:
        store.destroy()


def test_noalloc_rejects_oversize_requests():
    import torch
    from kv_cache_injection_gb300 import _lib, api
    gh.ensure_built()
    z64 = torch.zeros((1,), dtype=torch.int64, device="cuda")
    z32 = torch.zeros((1,), dtype=torch.int32, device="cuda")
    arena = torch.zeros((4, 1, 2, 4, 64), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((1, 2, 1, 16, 4, 64), dtype=torch.bfloat16, device="cuda")
    big = torch.zeros((_lib.IS_NOALLOC_MAX_REQUESTS + 1, 1), dtype=torch.int64, device="cuda")
    with pytest.raises(api.ISError) as e:
        api.is_inject_noalloc(arena, z64, z32, 4, 1, 4, 64, "bf16", big,
                              torch.zeros(big.shape[0], dtype=torch.int32, device="cuda"),
                              torch.zeros(big.shape[0], dtype=torch.int32, device="cuda"),
                              api.make_rope(1e4), torch.zeros((big.shape[0], 1), dtype=torch.int32,
                                                              device="cuda"),
                              api.make_cache_desc(16, 1, "bf16"), cache, z32)
    assert e.value.status == 8 and "IS_NOALLOC_MAX_REQUESTS" in str(e.value)
    wide = torch.zeros((1, _lib.IS_NOALLOC_MAX_FACTS + 1), dtype=torch.int64, device="cuda")
    with pytest.raises(api.ISError) as e:
        api.is_inject_noalloc(arena, z64, z32, 4, 1, 4, 64, "bf16", wide, z32, z32,
                              api.make_rope(1e4), torch.zeros((1, 1), dtype=torch.int32, device="cuda"),
                              api.make_cache_desc(16, 1, "bf16"), cache, z32)
    assert e.value.status == 8
