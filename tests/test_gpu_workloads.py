"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (the fused is_retrieve_and_inject).

At these sizes the oracle checks every query's top-k, every request's segment
length and every slot of the slot mapping; every cache row is checked on the
device to have changed exactly when its slot was targeted.  The injected
tokens are compared element by element with the oracle: all of them for the
single-request workloads (Llama-3.1-8B, the Mistral-7B k sweep, Qwen3-14B) and
for one Qwen2.5-7B user; a sample (first and last token of every segment plus
random ones, all layers and heads) for the other 99 users and for the capacity
workload's 320 000 tokens.
"""
import pytest

from synth import staging, workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    gh.ensure_built()
    from kv_cache_injection_gb300 import api as a
    return a


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
        st = gh.check_fused_workload(api, wl, store, all_tokens=True)
        assert st["tokens"] > 40 * 10
        assert st["n"] == st["tokens"] * wl.spec.token_elems      # every injected key element

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
        st = gh.check_fused_workload(api, wl, store, k=k, all_tokens=True)
        assert st["tokens"] >= 10 * k
        assert st["n"] == st["tokens"] * wl.spec.token_elems


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
        st = gh.check_fused_workload(api, wl, store, sample_tokens=300, all_tokens=[0])
        assert st["tokens"] > 100 * 50 * 10
        assert st["tokens_compared_in_full"] >= 50 * 10

    def test_fused_parity_tensor_core_similarity(self, api, loaded):
        """The same 100 queries with the similarity as tcgen05 contractions
        (one group per user), then the per-user top-k."""
        from kv_cache_injection_gb300 import _lib
        wl, store = loaded
        api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_BATCHED)
        try:
            st = gh.check_fused_workload(api, wl, store, sample_tokens=300, seed=1)
        finally:
            api.is_set_retrieval_mode(store, _lib.IS_RETRIEVAL_AUTO)
        assert st["tokens"] > 100 * 50 * 10


class TestQwen3_14B:
    """The larger model the pages scale to: Qwen3-14B KV shape, k = 50."""

    @pytest.fixture(scope="class")
    @classmethod
    def loaded(cls, api):
        wl = workloads.get("qwen3_14b")
        store = staging.load_store(wl, api)
        yield wl, store
        store.destroy()

    def test_fused_parity(self, api, loaded):
        wl, store = loaded
        st = gh.check_fused_workload(api, wl, store, all_tokens=True)
        assert st["tokens"] > 50 * 10
        assert st["n"] == st["tokens"] * wl.spec.token_elems


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
        st = gh.check_fused_workload(api, wl, store, sample_tokens=400)
        assert st["tokens"] > 64 * 200 * 4
