"""Seeded random configurations against the oracle, every injected token
compared: element type, pairing style and frequency scaling, layer count and
head shape, block size (1 to 64), fact lengths, k, number and mix of users,
segment starts, the store's placement and an FP8 cache.  Sizes stay small so
the oracle compares every row."""
import numpy as np
import pytest

from synth import staging, workloads
from tests import gpu_helpers as gh
from tests import parity

pytestmark = pytest.mark.gpu

N_CASES = 48


@pytest.fixture(scope="module")
def api():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api as a
    return a


def _case(i):
    rng = np.random.default_rng(1000 + i)
    dtype = ["f32", "bf16", "f16"][i % 3]
    elt = 4 if dtype == "f32" else 2
    style = int(rng.integers(0, 2))
    ve = 16 // elt
    max_d = 32 * ve * (2 if style == 0 else 1)           # widest head the kernels take
    D = int(rng.choice([d for d in (16, 32, 64, 128, 256, 512) if d <= max_d]))
    H = max(1, 512 // (D * elt)) * int(rng.choice([1, 2]))   # rows of a multiple of 512 bytes
    scaled = bool(rng.integers(0, 2))
    rope = (workloads.RopeSpec(theta=float(rng.choice([1e4, 5e5, 1e6])), style=style, scaling=1,
                               factor=float(rng.choice([4.0, 8.0])), low_freq_factor=1.0,
                               high_freq_factor=4.0, original_max_pos=int(rng.choice([64, 512, 8192])))
            if scaled else workloads.RopeSpec(theta=float(rng.choice([1e4, 5e5, 1e6])), style=style))
    n_users = int(rng.integers(1, 5))
    k = int(rng.choice([1, 3, 8, 17, 33, 64]))
    max_len = int(rng.choice([1, 4, 12, 30]))
    bs = int(rng.choice([1, 8, 16, 32, 64]))
    n_q = n_users if rng.integers(0, 2) else int(rng.integers(1, 9))
    share = n_q != n_users
    spec = workloads.WorkloadSpec(
        name=f"fuzz{i}", num_layers=int(rng.integers(1, 5)), num_kv_heads=H, head_dim=D, kv_dtype=dtype,
        rope=rope, n_users=n_users, facts_per_user=int(rng.integers(max(k // 2, 1), 400)),
        length_dist=("uniform", 1, max_len), emb_dim=int(rng.choice([64, 128, 256])),
        emb_dtype="f32" if dtype == "f32" else "f16", n_queries=n_q, k=k, query_kind="planted",
        start=("uniform", 0, int(rng.choice([1, 100, 5000, 100000]))), block_size=bs,
        tokens_cap=k * max_len, block_layout="free_list", queries_share_user=share, seed=2000 + i)
    placement = "host" if rng.integers(0, 4) == 0 else "device"
    fp8 = dtype != "f32" and rng.integers(0, 4) == 0
    scales = (float(rng.uniform(0.2, 2.0)), float(rng.uniform(0.2, 2.0)))
    return spec, placement, fp8, scales


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_configuration(api, i):
    spec, placement, fp8, scales = _case(i)
    wl = workloads.generate(spec)
    if spec.queries_share_user and spec.n_users > 1:
        wl.users[:] = np.random.default_rng(i).integers(0, spec.n_users, size=spec.n_queries).astype(np.int32)
    store = staging.load_store(wl, api, kv_placement=placement)
    try:
        n_tok = sum(len(pl) for pl in parity.oracle_plans(wl, [
            parity.oracle_retrieve(wl, q, spec.k)[0] for q in range(spec.n_queries)])[0])
        st = gh.check_fused_workload(api, wl, store, sample_tokens=max(n_tok, 1),
                                     cache_dtype="e4m3" if fp8 else None,
                                     k_scale=scales[0], v_scale=scales[1])
        assert st["tokens"] == n_tok
    finally:
        store.destroy()


def _batched_case(i):
    rng = np.random.default_rng(3000 + i)
    n_users = int(rng.integers(1, 5))
    per_user = [int(rng.integers(1, 151)) for _ in range(n_users)]
    users = np.concatenate([np.full(c, u, np.int32) for u, c in enumerate(per_user)])
    users = rng.permutation(users)[:1024]
    k = int(rng.choice([1, 7, 50, 100, 200]))
    spec = workloads.WorkloadSpec(
        name=f"fuzz_batched{i}", num_layers=1, num_kv_heads=4, head_dim=64, kv_dtype="bf16",
        rope=workloads.RopeSpec(theta=1e4), n_users=n_users, facts_per_user=int(rng.integers(64, 3000)),
        length_dist=("uniform", 1, 3), emb_dim=int(rng.choice([64, 72, 136, 200, 1024])), emb_dtype="f16",
        n_queries=len(users), k=k, query_kind="planted", start=("uniform", 0, 50), block_size=16,
        tokens_cap=k * 3, block_layout="free_list", queries_share_user=True, seed=4000 + i)
    return spec, users


@pytest.mark.parametrize("i", range(12))
def test_random_tensor_core_retrieval(api, i):
    """The tcgen05 similarity path on random embedding widths (not only
    multiples of the 64-element TMA chunk), users and group sizes (groups of
    at most 64 queries per user): top-k against the oracle, scores against the
    per-query path."""
    import torch
    from kv_cache_injection_gb300 import _lib
    spec, users = _batched_case(i)
    wl = workloads.generate(spec)
    wl.users[:] = users
    store = staging.load_store(wl, api)
    try:
        inp = staging.device_inputs(wl)
        Q, k = spec.n_queries, spec.k
        out = {}
        for mode in (_lib.IS_RETRIEVAL_BATCHED, _lib.IS_RETRIEVAL_PER_QUERY):
            api.is_set_retrieval_mode(store, mode)
            ids = torch.full((Q, k), -7, dtype=torch.int64, device="cuda")
            sc = torch.zeros((Q, k), dtype=torch.float32, device="cuda")
            api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
            assert api.is_get_status(store) == 0
            out[mode] = (ids.cpu().numpy(), sc.cpu().numpy())
        ids_b, sc_b = out[_lib.IS_RETRIEVAL_BATCHED]
        for q in range(Q):
            o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, k)
            parity.check_topk(ids_b[q], sc_b[q], o_ids, o_sc, score_of, k)
        assert np.max(np.abs(sc_b - out[_lib.IS_RETRIEVAL_PER_QUERY][1])) <= 2e-6
    finally:
        store.destroy()


@pytest.mark.parametrize("i", range(12))
def test_random_explicit_lists_and_layerwise(api, i):
    """is_inject with random explicit lists (empty requests, a fact repeated
    within and across requests, any order), then the same plan layer by layer
    through is_inject_layer into per-layer caches: every token against the
    oracle, every layer equal to the whole-cache injection."""
    import torch
    spec, placement, fp8, scales = _case(100 + i)
    rng = np.random.default_rng(5000 + i)
    wl = workloads.generate(spec.with_(n_users=1, queries_share_user=True))
    s = wl.spec
    store = staging.load_store(wl, api, kv_placement=placement)
    try:
        R, stride = s.n_queries, s.k
        n_ids = rng.integers(0, stride + 1, size=R).astype(np.int32)
        ids = np.full((R, stride), -1, dtype=np.int64)
        for r in range(R):
            ids[r, :n_ids[r]] = rng.integers(0, s.n_facts, size=n_ids[r])      # repeats allowed
        inp = staging.device_inputs(wl)
        cdt = "e4m3" if fp8 else None
        cache = staging.canary_cache(wl, cache_dtype=cdt)
        cd = api.make_cache_desc(s.block_size, cache.shape[2], cdt or s.kv_dtype, *scales)
        rope = staging.rope_params(wl, api)
        seg_len = torch.empty(R, dtype=torch.int32, device="cuda")
        slots = torch.full((R * stride * int(wl.lengths.max()) + 1,), -9, dtype=torch.int64, device="cuda")
        d_ids, d_n = torch.from_numpy(ids).cuda(), torch.from_numpy(n_ids).cuda()
        api.is_inject(store, d_ids, d_n, inp["seg_start"], rope, inp["block_table"], cd, cache,
                      users=inp["users"], seg_len_out=seg_len, slot_mapping_out=slots)
        assert api.is_get_status(store) == 0
        rows = [ids[r, :n_ids[r]] for r in range(R)]
        plans, lens = parity.oracle_plans(wl, rows)
        assert np.array_equal(seg_len.cpu().numpy(), lens)
        want = np.concatenate([[e[3] for e in pl] for pl in plans] + [[]]).astype(np.int64)
        assert np.array_equal(slots.cpu().numpy()[: len(want)], want)
        gh.assert_only_slots_changed(cache, cdt or s.kv_dtype, want)
        entries = [e for pl in plans for e in pl]
        if entries:
            gk, gv = gh.gather_rows(cache, [e[3] for e in entries])
            if fp8:
                parity.compare_tokens_fp8(wl, gk, gv, entries, parity.oracle_freqs(wl), s.rope.style,
                                          parity.FactCache(wl), *scales)
            else:
                parity.compare_tokens(wl, gk, gv, entries, parity.oracle_freqs(wl), s.rope.style,
                                      parity.FactCache(wl))
        # the same plan, layer by layer, into per-layer caches
        for layer in range(s.num_layers):
            lc = staging.canary_cache(wl, cache_dtype=cdt)[0].contiguous()
            if layer == 0:
                api.is_inject_layer(store, 0, R, inp["seg_start"], rope, inp["block_table"], cd, lc,
                                    fact_ids=d_ids, n_ids=d_n, users=inp["users"])
            else:
                api.is_inject_layer(store, layer, R, inp["seg_start"], rope, inp["block_table"], cd, lc)
            assert api.is_get_status(store) == 0
            assert torch.equal(lc.view(torch.uint8), cache[layer].contiguous().view(torch.uint8))
    finally:
        store.destroy()


@pytest.mark.parametrize("i", range(8))
def test_random_capture_equals_add_facts(api, i):
    """Context-Window Encoding capture with random windows and lengths (layer
    buffers with random content) stores exactly the fact rows: a store built
    by is_store_add_facts from those rows injects the same cache byte for byte."""
    import torch
    rng = np.random.default_rng(6000 + i)
    spec, placement, _, _ = _case(200 + i)
    L, H, D, dt = spec.num_layers, spec.num_kv_heads, spec.head_dim, spec.kv_dtype
    tdt = staging.torch_dtype(dt)
    n = int(rng.integers(1, 40))
    lengths = rng.integers(1, 20, size=n).astype(np.int32)
    windows = rng.integers(0, 50, size=n).astype(np.int32)
    total = int((lengths + windows).sum())
    gen = torch.Generator(device="cuda").manual_seed(i)
    layers = [(torch.randn(total, H, D, device="cuda", generator=gen).to(tdt),
               torch.randn(total, H, D, device="cuda", generator=gen).to(tdt)) for _ in range(L)]
    emb = torch.nn.functional.normalize(torch.randn(n, 64, device="cuda", generator=gen), dim=1)
    emb = emb.half() if spec.emb_dtype == "f16" else emb
    def store():
        cfg = api.make_config(num_layers=L, num_kv_heads=H, head_dim=D, emb_dim=64, kv_dtype=dt,
                              emb_dtype=spec.emb_dtype, max_facts=n, max_tokens=int(lengths.sum()),
                              max_users=1, max_queries=1, max_k=n, max_requests=1, kv_placement=placement)
        return api.is_store_create(cfg, 0)
    a, b = store(), store()
    try:
        api.is_store_capture_begin(a, 0, windows, lengths, emb)
        for l in rng.permutation(L):
            api.is_store_capture_layer(a, int(l), layers[l][0], layers[l][1])
        assert np.array_equal(api.is_store_capture_end(a, n), np.arange(n))
        # the fact rows, token-major [tokens][L][H][D]
        starts = np.cumsum(np.concatenate([[0], lengths + windows]))[:-1] + windows
        idx = torch.from_numpy(np.concatenate([np.arange(st, st + ln) for st, ln in zip(starts, lengths)])).cuda()
        k = torch.stack([layers[l][0].index_select(0, idx) for l in range(L)], 1).contiguous()
        v = torch.stack([layers[l][1].index_select(0, idx) for l in range(L)], 1).contiguous()
        api.is_store_add_facts(b, 0, lengths, k, v, emb)
        bs = 16
        T = int(lengths.sum())
        nb = T // bs + 2
        bt = torch.arange(nb, dtype=torch.int32, device="cuda")[None].flip(1).contiguous()
        rope = api.make_rope(1e4, spec.rope.style)
        cd = api.make_cache_desc(bs, nb, dt)
        order = torch.from_numpy(rng.permutation(n).astype(np.int64)[None]).cuda()
        outs = []
        for st in (a, b):
            cache = torch.zeros((L, 2, nb, bs, H, D), dtype=tdt, device="cuda")
            api.is_inject(st, order, torch.tensor([n], dtype=torch.int32, device="cuda"),
                          torch.zeros(1, dtype=torch.int32, device="cuda"), rope, bt, cd, cache)
            assert api.is_get_status(st) == 0
            outs.append(cache)
        assert torch.equal(outs[0].view(torch.uint8), outs[1].view(torch.uint8))
    finally:
        a.destroy()
        b.destroy()


def _topk_case(i):
    rng = np.random.default_rng(5000 + i)
    n_users = int(rng.integers(1, 4))
    n = int(rng.choice([int(rng.integers(1, 300)), int(rng.integers(1500, 2600)), int(rng.integers(3900, 6200))]))
    k = int(rng.choice([1, 5, 50, 64, 65, 200, 257, 1024]))
    n_q = int(rng.integers(1, 9))
    spec = workloads.WorkloadSpec(
        name=f"fuzz_topk{i}", num_layers=1, num_kv_heads=4, head_dim=64, kv_dtype="bf16",
        rope=workloads.RopeSpec(theta=1e4), n_users=n_users, facts_per_user=n,
        length_dist=("uniform", 1, 2), emb_dim=int(rng.choice([64, 128, 1024])), emb_dtype="f16",
        n_queries=n_q, k=min(k, 1024), query_kind="planted", start=("uniform", 0, 50), block_size=16,
        tokens_cap=64, block_layout="free_list", queries_share_user=True, seed=6000 + i)
    dup = int(rng.choice([0, 0, 3, 40]))        # embeddings drawn from this many distinct rows (0: all distinct)
    return spec, rng, dup


@pytest.mark.parametrize("i", range(24))
def test_random_topk(api, i):
    """Retrieval alone on random user sizes either side of the kernels' internal
    limits (2048 rows for bins counted by the similarity CTAs, 4096 for keys
    staged in shared memory), k across the rank (<= 256 candidates), bitonic and
    radix-select paths, several queries and, in some draws, many exact ties
    (embeddings repeated).  Per-query path, every top-k against the oracle."""
    import torch
    from kv_cache_injection_gb300 import _lib
    spec, rng, dup = _topk_case(i)
    wl = workloads.generate(spec)
    wl.users[:] = rng.integers(0, spec.n_users, size=spec.n_queries).astype(np.int32)
    dup = min(dup, len(wl.emb))
    if dup:
        base = wl.emb[:dup].copy()
        wl.emb[:] = base[rng.integers(0, dup, size=len(wl.emb))]
        wl.queries[:] = base[rng.integers(0, dup, size=len(wl.queries))]
    store = staging.load_store(wl, api, max_k=1024)
    try:
        api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_PER_QUERY)
        inp = staging.device_inputs(wl)
        k = spec.k
        for rep in range(2):                    # twice: the bins must be left zeroed
            ids = torch.empty((spec.n_queries, k), dtype=torch.int64, device="cuda")
            sc = torch.empty((spec.n_queries, k), dtype=torch.float32, device="cuda")
            api.is_retrieve_topk(store, inp["users"], inp["q_emb"], k, ids, sc)
            g, gs = ids.cpu().numpy(), sc.cpu().numpy()
            for q in range(spec.n_queries):
                o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, k)
                parity.check_topk(g[q], gs[q], o_ids, o_sc, score_of, k)
        assert api.is_get_status(store) == 0
    finally:
        store.destroy()
