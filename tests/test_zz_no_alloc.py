"""The allocation-free entry point, is_inject_noalloc.

Some callers cannot allocate device memory: a serving engine that reserves
all of HBM for its own pools at start-up and hands kernels only memory it
owns, or code running where cudaMalloc is not allowed.  is_inject_noalloc
serves them: the caller keeps the facts' pre-RoPE K and raw V in its own
token-major buffer and passes inputs and outputs; the library creates no store
and keeps the per-request segment plan in a fixed static device array.

The tests call it through the C ABI:
* twice in a row on a small shape (two request batches on one stream, so the
  second call overwrites the static array the first used): each output is
  compared with the existing is_inject entry point on a store holding the same
  facts (values bit for bit, rotated keys within one bf16 ulp, segment lengths
  and slot mappings exactly) and, every injected token, with the oracle;
* three times in a row on the Llama-3.1-8B KV shape with 256 facts per call,
  enough work that the inject kernel hands out part of it through the static
  array's chunk counters: each call against is_inject over the whole cache and
  against the oracle (every token of the first call, a sample of the others);
* with host-made bad rows in the caller's fact table (a length of 0, a length
  past max_fact_len, a negative first token, a fact running past the arena):
  the status bit is latched, those facts are left out, every other fact is
  injected as the oracle says and every other cache row keeps its canary;
* with requests past the static array's limits, which are refused before
  anything is enqueued.
It lives in a file of its own that pytest collects last.
"""
import numpy as np
import pytest

from synth import kvgen, staging, workloads
from tests import gpu_helpers as gh
from tests import parity

pytestmark = pytest.mark.gpu

SPEC = workloads.WorkloadSpec(
    name="noalloc_bf16", num_layers=3, num_kv_heads=4, head_dim=64, kv_dtype="bf16",
    rope=workloads.RopeSpec(theta=5e5, scaling=1, factor=8.0, low_freq_factor=1.0,
                            high_freq_factor=4.0, original_max_pos=64),
    n_users=1, facts_per_user=300, length_dist=("uniform", 1, 21), emb_dim=64, emb_dtype="f16",
    n_queries=6, k=12, query_kind="planted", start=("uniform", 0, 500), block_size=16,
    tokens_cap=12 * 21, block_layout="free_list", queries_share_user=True, seed=31)

# Llama-3.1-8B KV shape (32 layers, 8 KV heads of 128, bf16); 8 requests of 32 facts.
POOL_SPEC = workloads.WorkloadSpec(
    name="noalloc_llama", num_layers=32, num_kv_heads=8, head_dim=128, kv_dtype="bf16",
    rope=workloads.LLAMA31_ROPE, n_users=1, facts_per_user=400, length_dist=("uniform", 10, 40),
    emb_dim=64, emb_dtype="f16", n_queries=8, k=32, query_kind="planted", start=("uniform", 0, 3000),
    block_size=16, tokens_cap=32 * 40, block_layout="free_list", queries_share_user=True, seed=33)

IS_ST_FACT_RANGE = 0x01


def _requests(wl, seed, full=False):
    rng = np.random.default_rng(seed)
    R, stride = wl.spec.n_queries, wl.spec.k
    n_ids = (np.full(R, stride) if full else rng.integers(0, stride + 1, size=R)).astype(np.int32)
    ids = np.full((R, stride), -1, dtype=np.int64)
    for r in range(R):
        ids[r, :n_ids[r]] = rng.choice(wl.spec.n_facts, size=n_ids[r], replace=False)
    return ids, n_ids


class Caller:
    """A caller's own buffers: the token-major arena [T][L][2][H][D] with the
    workload's facts, its fact table, and a store holding the same facts for
    the is_inject reference."""

    def __init__(self, api, wl):
        import torch
        s = wl.spec
        self.api, self.wl = api, wl
        self.store = staging.load_store(wl, api)
        T = wl.total_tokens
        k = torch.empty((T, s.num_layers, s.num_kv_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
        v = torch.empty_like(k)
        staging.fill_kv(k, "bf16", s.seed, kvgen.STREAM_K, 0)
        staging.fill_kv(v, "bf16", s.seed, kvgen.STREAM_V, 0)
        self.arena = torch.stack([k, v], dim=2).contiguous()
        del k, v
        self.fact_tok = torch.from_numpy(wl.tok_base).cuda()
        self.fact_len = torch.from_numpy(wl.lengths).cuda()
        self.inp = staging.device_inputs(wl)
        self.rope = staging.rope_params(wl, api)
        self.cdesc = api.make_cache_desc(s.block_size, wl.num_blocks, "bf16")
        self.max_len = int(wl.lengths.max())

    def noalloc(self, d_ids, d_n, status, fact_tok=None, fact_len=None):
        import torch
        s = self.wl.spec
        cache = staging.canary_cache(self.wl)
        seg_len = torch.full((s.n_queries,), -1, dtype=torch.int32, device="cuda")
        slots = torch.full((s.n_queries * s.k * self.max_len,), -9, dtype=torch.int64, device="cuda")
        self.api.is_inject_noalloc(
            self.arena, self.wl.total_tokens, self.fact_tok if fact_tok is None else fact_tok,
            self.fact_len if fact_len is None else fact_len, self.max_len, s.num_layers,
            s.num_kv_heads, s.head_dim, "bf16", d_ids, d_n, self.inp["seg_start"], self.rope,
            self.inp["block_table"], self.cdesc, cache, status, seg_len_out=seg_len, slot_mapping_out=slots)
        return cache, seg_len, slots

    def reference(self, d_ids, d_n, seg_len_like, slots_like):
        import torch
        ref = staging.canary_cache(self.wl)
        ref_len = torch.full_like(seg_len_like, -1)
        ref_slots = torch.full_like(slots_like, -9)
        self.api.is_inject(self.store, d_ids, d_n, self.inp["seg_start"], self.rope, self.inp["block_table"],
                           self.cdesc, ref, seg_len_out=ref_len, slot_mapping_out=ref_slots)
        assert self.api.is_get_status(self.store) == 0
        return ref, ref_len, ref_slots


def _assert_same_as_is_inject(out, ref):
    """Segment lengths and slots exactly; values and untouched rows bit for
    bit; rotated keys within one bf16 ulp (compared on the device, so the
    whole cache is checked)."""
    import torch
    from oracle import numerics
    (cache, seg_len, slots), (rc, r_len, r_slots) = out, ref
    assert torch.equal(seg_len, r_len) and int(seg_len.sum()) > 0
    assert torch.equal(slots, r_slots)
    a, b = cache.view(torch.int16), rc.view(torch.int16)
    assert torch.equal(a[:, 1], b[:, 1])                               # V and untouched rows
    diff = a[:, 0] != b[:, 0]
    if bool(diff.any()):
        ga = staging.cache_bits(cache[:, 0][diff]).astype(np.uint16)
        gb = staging.cache_bits(rc[:, 0][diff]).astype(np.uint16)
        da, db = numerics.decode(ga, "bf16"), numerics.decode(gb, "bf16")
        assert np.all(np.abs(da - db) <= numerics.ulp(db, "bf16"))


def _assert_matches_oracle(wl, out, ids, sample=None, seed=0):
    """The call's output against the oracle: segment lengths, slots and
    canaries exactly; the injected tokens (all of them, or first and last of
    each segment plus ``sample`` random ones) element by element."""
    cache, seg_len, slots = out
    plans, lens = parity.oracle_plans(wl, ids)
    assert np.array_equal(seg_len.cpu().numpy(), lens)
    want = np.concatenate([[e[3] for e in pl] for pl in plans]).astype(np.int64)
    assert np.array_equal(slots.cpu().numpy()[: len(want)], want)
    gh.assert_only_slots_changed(cache, "bf16", want)
    entries = [e for pl in plans for e in pl]
    if sample is not None:
        rng = np.random.default_rng(seed)
        pick = set(rng.choice(len(entries), size=min(sample, len(entries)), replace=False).tolist())
        off = 0
        for pl in plans:
            if pl:
                pick.update([off, off + len(pl) - 1])
            off += len(pl)
        entries = [entries[i] for i in sorted(pick)]
    gk, gv = gh.gather_rows(cache, [e[3] for e in entries])
    st = parity.compare_runs(wl, gk, gv, entries, parity.oracle_freqs(wl), wl.spec.rope.style,
                             gh.DeviceFactCache(wl))
    assert st["n"] == len(entries) * wl.spec.token_elems
    return st


@pytest.fixture(scope="module")
def small():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api
    c = Caller(api, workloads.generate(SPEC))
    yield c
    c.store.destroy()


def test_noalloc_matches_is_inject_on_two_calls_in_a_row(small):
    import torch
    c = small
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    calls = []
    for seed in (1, 2):                       # two calls in a row, same stream
        ids, n_ids = _requests(c.wl, seed)
        d_ids, d_n = torch.from_numpy(ids).cuda(), torch.from_numpy(n_ids).cuda()
        calls.append((ids, d_ids, d_n, c.noalloc(d_ids, d_n, status)))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for ids, d_ids, d_n, out in calls:
        _assert_same_as_is_inject(out, c.reference(d_ids, d_n, out[1], out[2]))
        _assert_matches_oracle(c.wl, out, ids)


def test_noalloc_bad_fact_rows_are_left_out(small):
    """Host-made bad rows of the caller's fact table; the device finds them."""
    import torch
    c = small
    wl = c.wl
    T = wl.total_tokens
    fact_tok = wl.tok_base.copy()
    fact_len = wl.lengths.copy()
    long_facts = np.nonzero(wl.lengths >= 2)[0]
    bad = {int(long_facts[0]): "len0", int(long_facts[1]): "len_big", int(long_facts[2]): "tok_neg",
           int(long_facts[3]): "past_end"}
    for f, kind in bad.items():
        if kind == "len0":
            fact_len[f] = 0
        elif kind == "len_big":
            fact_len[f] = c.max_len + 3
        elif kind == "tok_neg":
            fact_tok[f] = -5
        else:
            fact_tok[f] = T - 1
    good = [f for f in range(wl.spec.n_facts) if f not in bad][:40]
    R, stride = wl.spec.n_queries, wl.spec.k
    ids = np.full((R, stride), -1, dtype=np.int64)
    n_ids = np.zeros(R, dtype=np.int32)
    rng = np.random.default_rng(5)
    bad_list = list(bad)
    for r in range(R):
        row = list(rng.choice(good, size=stride - 2, replace=False)) + [bad_list[r % 4], bad_list[(r + 1) % 4]]
        rng.shuffle(row)
        ids[r] = row
        n_ids[r] = stride
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_ids, d_n = torch.from_numpy(ids).cuda(), torch.from_numpy(n_ids).cuda()
    out = c.noalloc(d_ids, d_n, status, torch.from_numpy(fact_tok).cuda(), torch.from_numpy(fact_len).cuda())
    torch.cuda.synchronize()
    assert int(status.item()) == IS_ST_FACT_RANGE
    # what the oracle injects once the bad facts are left out (a fact of length 0 adds nothing)
    _assert_matches_oracle(wl, out, np.where(np.isin(ids, bad_list), -1, ids))


@pytest.fixture(scope="module")
def pool():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api
    c = Caller(api, workloads.generate(POOL_SPEC))
    yield c
    c.store.destroy()


def test_noalloc_three_calls_through_the_chunk_pool(pool):
    """Launches large enough for the inject kernel's chunk pool (about 8000
    segment tokens x 32 layers over the persistent grid's warps), three in a
    row: every call starts from counters its own planning kernel zeroed."""
    import torch
    c = pool
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i, seed in enumerate((11, 12, 13)):
        ids, n_ids = _requests(c.wl, seed, full=True)
        d_ids, d_n = torch.from_numpy(ids).cuda(), torch.from_numpy(n_ids).cuda()
        out = c.noalloc(d_ids, d_n, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # work items (token, layer): the persistent grid has 2 CTAs of 8 warps
        # per SM, and each warp's static half-share is far past the 4 items
        # below which the kernel splits evenly and uses no pool
        items = int(out[1].sum()) * c.wl.spec.num_layers
        n_warps = 2 * 8 * torch.cuda.get_device_properties(0).multi_processor_count
        assert items // 2 // n_warps >= 16
        _assert_same_as_is_inject(out, c.reference(d_ids, d_n, out[1], out[2]))
        _assert_matches_oracle(c.wl, out, ids, sample=None if i == 0 else 200, seed=seed)
        del out


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
        api.is_inject_noalloc(arena, 4, z64, z32, 4, 1, 4, 64, "bf16", big,
                              torch.zeros(big.shape[0], dtype=torch.int32, device="cuda"),
                              torch.zeros(big.shape[0], dtype=torch.int32, device="cuda"),
                              api.make_rope(1e4), torch.zeros((big.shape[0], 1), dtype=torch.int32,
                                                              device="cuda"),
                              api.make_cache_desc(16, 1, "bf16"), cache, z32)
    assert e.value.status == 8 and "IS_NOALLOC_MAX_REQUESTS" in str(e.value)
    wide = torch.zeros((1, _lib.IS_NOALLOC_MAX_FACTS + 1), dtype=torch.int64, device="cuda")
    with pytest.raises(api.ISError) as e:
        api.is_inject_noalloc(arena, 4, z64, z32, 4, 1, 4, 64, "bf16", wide, z32, z32,
                              api.make_rope(1e4), torch.zeros((1, 1), dtype=torch.int32, device="cuda"),
                              api.make_cache_desc(16, 1, "bf16"), cache, z32)
    assert e.value.status == 8
    with pytest.raises(api.ISError) as e:                  # an empty arena
        api.is_inject_noalloc(arena, 0, z64, z32, 4, 1, 4, 64, "bf16", z64.view(1, 1), z32, z32,
                              api.make_rope(1e4), torch.zeros((1, 1), dtype=torch.int32, device="cuda"),
                              api.make_cache_desc(16, 1, "bf16"), cache, z32)
    assert e.value.status == 1
