"""The comparison helpers the GPU parity tests use, checked on the CPU.

A cache filled by the oracle itself must pass both the per-token and the
run-grouped comparisons with the same element counts, and one flipped bit in
a key or a value must fail them.
"""
import numpy as np
import pytest

from oracle import inject as oinject
from synth import workloads
from tests import parity


def _oracle_cache(wl, ids, dtype):
    s = wl.spec
    cache = np.empty(workloads.cache_shape(s, wl.num_blocks), dtype={"f32": np.float32}.get(dtype, np.uint16))
    cache[...] = np.asarray(workloads.CANARY_BITS[dtype]).astype(cache.dtype) if dtype != "f32" else np.nan
    facts = parity.FactCache(wl)
    oinject.inject(cache, dtype, facts, ids, wl.lengths, int(wl.seg_start[0]), wl.block_table[0],
                   s.block_size, parity.oracle_freqs(wl), s.rope.style)
    return cache, facts


def _gather(cache, slots):
    L, _, NB, bs, H, D = cache.shape
    flat = cache.reshape(L, 2, NB * bs, H, D)
    rows = flat[:, :, np.asarray(slots)].transpose(2, 0, 1, 3, 4)          # [n][L][2][H][D]
    return rows[:, :, 0].copy(), rows[:, :, 1].copy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_runs_equal_per_token_and_catch_errors(dtype):
    wl = workloads.get("tiny", kv_dtype=dtype)
    ids = [5, 17, 5, 3]                                       # a repeated fact makes two runs of it
    cache, facts = _oracle_cache(wl, ids, wl.spec.kv_dtype)
    plans, _ = parity.oracle_plans(wl, [ids])
    entries = plans[0]
    assert len(list(parity.fact_runs(entries))) == 4
    gk, gv = _gather(cache, [e[3] for e in entries])
    freqs, style = parity.oracle_freqs(wl), wl.spec.rope.style
    a = parity.compare_tokens(wl, gk, gv, entries, freqs, style, facts)
    b = parity.compare_runs(wl, gk, gv, entries, freqs, style, facts)
    assert a["n"] == b["n"] == len(entries) * wl.spec.token_elems
    assert a["within_1ulp"] == b["within_1ulp"]
    bad_k = gk.copy()
    bad_k[len(entries) // 2, 0, 1, 7:9].view(np.uint32)[0] ^= 1 << 20
    with pytest.raises(AssertionError):
        parity.compare_runs(wl, bad_k, gv, entries, freqs, style, facts)
    bad_v = gv.copy()
    bad_v[-1, 0, 0, 0:2].view(np.uint32)[0] ^= 1
    with pytest.raises(AssertionError):
        parity.compare_runs(wl, gk, bad_v, entries, freqs, style, facts)
