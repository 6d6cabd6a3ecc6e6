"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (the fused is_retrieve_and_inject).

At these sizes the oracle checks every query's top-k, every request's segment
length and every slot of the slot mapping, and rotates/compares a sample of
the injected tokens (all layers and heads of the sampled tokens); every
cache row is checked on the device to have changed exactly when its slot was
targeted.
"""
import numpy as np
import pytest

from synth import staging, workloads
from tests import gpu_helpers as gh
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api as a
    return a


def _check_workload(api, wl, store, k=None, sample_tokens=160, seed=0):
    inp = staging.device_inputs(wl)
    cache = staging.canary_cache(wl)
    k = wl.spec.k if k is None else k
    out = gh.run_fused(api, store, wl, inp, cache, k=k)
    assert out["status"] == 0, hex(out["status"])
    swapped = 0
    for q in range(wl.spec.n_queries):
        o_ids, o_sc, score_of = parity.oracle_retrieve(wl, q, k)
        swapped += parity.check_topk(out["ids"][q], out["scores"][q], o_ids, o_sc, score_of, k)["swapped"]
    plans, lens = parity.oracle_plans(wl, out["ids"])
    assert np.array_equal(out["seg_len"], lens)
    want_slots = np.concatenate([[e[3] for e in pl] for pl in plans]).astype(np.int64)
    assert np.array_equal(out["slot_map"][: len(want_slots)], want_slots)
    assert len(np.unique(want_slots)) == len(want_slots)
    gh.assert_only_slots_changed(cache, wl.spec.kv_dtype, want_slots)
    # sampled tokens: first and last token of every segment, plus random ones
    entries = [e for pl in plans for e in pl]
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(len(entries), size=min(sample_tokens, len(entries)), replace=False).tolist())
    off = 0
    for pl in plans:
        if pl:
            pick.update([off, off + len(pl) - 1])
        off += len(pl)
    sample = [entries[i] for i in sorted(pick)]
    gk, gv = gh.gather_rows(cache, [e[3] for e in sample])
    stats = parity.compare_tokens(wl, gk, gv, sample, parity.oracle_freqs(wl), wl.spec.rope.style,
                                  parity.FactCache(wl))
    del cache
    return {"tokens": int(lens.sum()), "swapped": swapped, **stats}


class TestLlama31:
    @pytest.fixture(scope="class")
    @classmethod
    def loaded(cls, api):
        wl = workloads.get("llama31_8b")
        store = staging.load_store(wl, api)
        yield wl, store
        store.destroy()

    def test_fused_parity(self, api, loaded):
        wl, store = loaded
        st = _check_workload(api, wl, store)
        assert st["tokens"] > 40 * 10

    def test_planted_fact_is_retrieved(self, api, loaded):
        import torch
        wl, store = loaded
        inp = staging.device_inputs(wl)
        ids = torch.empty((1, 50), dtype=torch.int64, device="cuda")
        sc = torch.empty((1, 50), dtype=torch.float32, device="cuda")
        api.is_retrieve_topk(store, inp["users"], inp["q_emb"], 50, ids, sc)
        assert int(ids[0, 0]) == int(wl.planted[0])


class TestMistralKSweep:
    @pytest.fixture(scope="class")
    @classmethod
    def loaded(cls, api):
        wl = workloads.get("mistral_7b")
        store = staging.load_store(wl, api)
        yield wl, store
        store.destroy()

    @pytest.mark.parametrize("k", [5, 10, 20, 50])
    def test_k(self, api, loaded, k):
        wl, store = loaded
        st = _check_workload(api, wl, store, k=k, sample_tokens=60, seed=k)
        assert st["tokens"] >= 10 * k


class TestQwen100Users:
    @pytest.fixture(scope="class")
    @classmethod
    def loaded(cls, api):
        wl = workloads.get("qwen25_7b_100u")
        store = staging.load_store(wl, api)
        yield wl, store
        store.destroy()

    def test_fused_parity(self, api, loaded):
        wl, store = loaded
        st = _check_workload(api, wl, store, sample_tokens=300)
        assert st["tokens"] > 100 * 50 * 10


@pytest.mark.slow
class TestCapacity:
    @pytest.fixture(scope="class")
    @classmethod
    def loaded(cls, api):
        wl = workloads.get("capacity")
        store = staging.load_store(wl, api, chunk_bytes=4 << 30)
        yield wl, store
        store.destroy()

    def test_fused_parity(self, api, loaded):
        wl, store = loaded
        info = api.is_store_info(store)
        assert info["n_tokens"] == wl.total_tokens and info["kv_bytes"] > 90e9
        st = _check_workload(api, wl, store, sample_tokens=400)
        assert st["tokens"] > 64 * 200 * 4
