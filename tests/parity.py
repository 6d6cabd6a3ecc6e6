"""Comparisons between the CUDA path and the fp64 oracle.

Tolerances (the method is exact, so these only absorb rounding):
* V copies, slot mappings, segment lengths, block placement: bit-exact;
* top-k: the id sets are equal except that ids whose oracle score lies within
  1e-4 of the k-th oracle score may be exchanged; every returned fp32 score is
  within 1e-5 of the oracle's fp64 cosine for that id; the order is checked
  wherever adjacent oracle scores differ by more than 1e-4;
* rotated keys, bf16: |g - o| <= 1 bf16 ulp of o, or |g - o| <= 2^-20 (|a| + |b|)
  where (a, b) is the rotated pair (the fp32-arithmetic floor near
  cancellation, where the ulp of the result is far below the inputs');
* rotated keys, fp32: |g - o| <= 4 ulp_f32(o) + 2^-22 (|a| + |b|);
* FP8 E4M3 cache (x stored as E4M3(x * r), r = fp32(1 / scale)): V bytes
  bit-exact against the oracle's fp32 product; keys |g - t| <= 1 E4M3 ulp of
  t = o * r, or 2^-20 (|a| + |b|) r near cancellation, and exactly +-448 where
  |t| > 448 (saturation).
"""
from __future__ import annotations

import numpy as np

from oracle import inject as oinject
from oracle import numerics, retrieval, rope
from synth import kvgen
from synth.workloads import CANARY_BITS

TIE_TOL = 1e-4
SCORE_TOL = 1e-5


def oracle_retrieve(wl, q: int, k: int):
    facts = wl.user_facts(int(wl.users[q]))
    scores = retrieval.cosine_scores(wl.queries[q].astype(np.float64), wl.emb[facts].astype(np.float64))
    ids, sc = retrieval.topk(scores, facts, k)
    return ids, sc, dict(zip(facts.tolist(), scores.tolist()))


def check_topk(gpu_ids, gpu_scores, o_ids, o_scores, score_of, k: int) -> dict:
    n = len(o_ids)
    gpu_ids = np.asarray(gpu_ids)
    gpu_scores = np.asarray(gpu_scores, dtype=np.float64)
    assert np.all(gpu_ids[n:] == -1), "rows beyond the user's facts must be -1"
    assert np.all(np.isneginf(gpu_scores[n:]))
    g = gpu_ids[:n]
    assert len(set(g.tolist())) == n, "duplicate ids"
    for i, s in zip(g.tolist(), gpu_scores[:n].tolist()):
        assert i in score_of, f"id {i} is not a fact of this user"
        assert abs(s - score_of[i]) <= SCORE_TOL, (i, s, score_of[i])
    so, sg = set(o_ids.tolist()), set(g.tolist())
    swapped = so ^ sg
    if n < k:
        assert not swapped, "a user with fewer than k facts returns all of them"
    kth = float(o_scores[n - 1]) if n else 0.0
    for i in swapped:
        assert abs(score_of[i] - kth) <= TIE_TOL, f"id {i} (score {score_of[i]}) vs k-th {kth}"
    for a, b in zip(g[:-1].tolist(), g[1:].tolist()):
        assert score_of[a] >= score_of[b] - TIE_TOL, "order"
    return {"swapped": len(swapped) // 2}


def partner_index(D: int, style: int) -> np.ndarray:
    i = np.arange(D)
    return i ^ (D // 2) if style == 0 else i ^ 1


def check_rotated(g_enc, o_f64, x_f64, style: int, dtype: str) -> dict:
    """g_enc: GPU rows in storage encoding; o_f64: oracle rotated rows; x_f64:
    the pre-RoPE rows (for the pair magnitudes).  Last axis is head_dim."""
    g = numerics.decode(g_enc, dtype)
    D = g.shape[-1]
    mag = np.abs(x_f64) + np.abs(x_f64[..., partner_index(D, style)])
    diff = np.abs(g - o_f64)
    if dtype == "f32":
        ok = diff <= 4 * numerics.ulp(o_f64, "f32") + 2.0 ** -22 * mag
        within_ulp = ok
    else:
        within_ulp = diff <= numerics.ulp(o_f64, dtype)
        ok = within_ulp | (diff <= 2.0 ** -20 * mag)
    bad = np.argwhere(~ok)
    assert bad.size == 0, (f"{len(bad)} rotated elements out of tolerance, first at {bad[0]}: "
                           f"gpu {g[tuple(bad[0])]!r} oracle {o_f64[tuple(bad[0])]!r}")
    return {"n": int(diff.size), "within_1ulp": int(within_ulp.sum()),
            "floor_only": int((ok & ~within_ulp).sum())}


class FactCache:
    """Oracle-side K/V, regenerated from the generator definition: whole facts
    (``cache(f)``) or single tokens (``cache.token(f, t)``)."""

    def __init__(self, wl):
        self.wl = wl
        self._m = {}

    def __call__(self, f: int):
        f = int(f)
        if f not in self._m:
            self._m[f] = (self.wl.fact_kv(f, kvgen.STREAM_K), self.wl.fact_kv(f, kvgen.STREAM_V))
        return self._m[f]

    def token(self, f: int, t: int):
        f, t = int(f), int(t)
        if f in self._m:
            return self._m[f][0][t], self._m[f][1][t]
        return self.wl.token_kv(f, t, kvgen.STREAM_K), self.wl.token_kv(f, t, kvgen.STREAM_V)


def oracle_plans(wl, ids_rows):
    """Per request: list of (fact, t, p, slot) following the oracle's composition."""
    bs = wl.spec.block_size
    plans, lens = [], []
    for r, ids in enumerate(ids_rows):
        plan, T = oinject.compose([int(i) for i in ids if i >= 0], wl.lengths, int(wl.seg_start[r]))
        plans.append([(f, j, p, oinject.slot(p, wl.block_table[r], bs)) for f, j, p in plan])
        lens.append(T)
    return plans, np.asarray(lens, dtype=np.int64)


def compare_tokens(wl, gathered_k, gathered_v, entries, freqs, style: int, facts: FactCache) -> dict:
    """gathered_k/v: [n][L][H][D] GPU cache rows (storage encoding) at the
    slots of ``entries`` = list of (fact, t, p, slot)."""
    dtype = wl.spec.kv_dtype
    stats = {"n": 0, "within_1ulp": 0, "floor_only": 0}
    for i, (f, j, p, _) in enumerate(entries):
        Kj, Vj = facts.token(f, j)
        assert np.array_equal(np.asarray(gathered_v[i]).view(np.uint8), Vj.view(np.uint8)), \
            f"V of fact {f} token {j} differs"
        x = numerics.decode(Kj, dtype)
        o = oinject.rotated_key_rows(Kj, p, freqs, style, dtype)
        st = check_rotated(gathered_k[i], o, x, style, dtype)
        for key in stats:
            stats[key] += st[key]
    return stats


def fact_runs(entries):
    """Split plan entries (fact, t, p, slot) into runs of consecutive tokens of
    one fact: yields (i0, i1, fact, t array, p array)."""
    i = 0
    while i < len(entries):
        f, t0 = entries[i][0], entries[i][1]
        j = i + 1
        while j < len(entries) and entries[j][0] == f and entries[j][1] == t0 + (j - i):
            j += 1
        yield (i, j, int(f), np.array([e[1] for e in entries[i:j]]),
               np.array([e[2] for e in entries[i:j]], dtype=np.int64))
        i = j


def compare_runs(wl, gathered_k, gathered_v, entries, freqs, style: int, facts,
                 fp8_scales=None) -> dict:
    """compare_tokens (or compare_tokens_fp8 when ``fp8_scales`` = (k_scale,
    v_scale)) over every entry, one fact run at a time: the same checks,
    vectorised over the run's tokens.  ``facts(f)`` returns the whole fact's
    (K, V) [len][L][H][D] in storage encoding."""
    dtype = wl.spec.kv_dtype
    stats = {"n": 0, "within_1ulp": 0, "floor_only": 0, "saturated": 0, "v_saturated": 0}
    for i0, i1, f, ts, ps in fact_runs(entries):
        K, V = facts(f)
        Kt, Vt = K[ts], V[ts]
        o = oinject.rotated_key_rows(Kt, ps[:, None, None], freqs, style, dtype)
        x = numerics.decode(Kt, dtype)
        if fp8_scales is None:
            assert np.array_equal(np.asarray(gathered_v[i0:i1]).view(np.uint8), Vt.view(np.uint8)), \
                f"V of fact {f} differs"
            st = check_rotated(gathered_k[i0:i1], o, x, style, dtype)
        else:
            k_scale, v_scale = fp8_scales
            want_v = oinject.e4m3_value(Vt, dtype, v_scale)
            assert np.array_equal(np.asarray(gathered_v[i0:i1]), want_v), f"FP8 V of fact {f} differs"
            stats["v_saturated"] += int((np.abs(numerics.e4m3_bits_to_f64(want_v)) == numerics.E4M3_MAX).sum())
            st = check_rotated_e4m3(gathered_k[i0:i1], o, x, style, k_scale)
        for key, val in st.items():
            stats[key] += val
    return stats


def oracle_freqs(wl):
    r = wl.spec.rope
    return rope.inv_freq(wl.spec.head_dim, r.theta, r.scaling, r.factor, r.low_freq_factor,
                         r.high_freq_factor, r.original_max_pos)


def canary_value(dtype: str):
    return CANARY_BITS[dtype]


def check_rotated_e4m3(g_bits, o_f64, x_f64, style: int, k_scale: float) -> dict:
    """Keys in an E4M3 cache against the oracle's fp64 rotation o."""
    r = float(oinject.scale_reciprocal(k_scale))
    g = numerics.e4m3_bits_to_f64(g_bits)
    t = o_f64 * r
    D = g.shape[-1]
    mag = (np.abs(x_f64) + np.abs(x_f64[..., partner_index(D, style)])) * r
    sat = np.abs(t) > numerics.E4M3_MAX
    within = np.abs(g - t) <= numerics.ulp(t, "e4m3")
    ok = np.where(sat, g == np.sign(t) * numerics.E4M3_MAX, within | (np.abs(g - t) <= 2.0 ** -20 * mag))
    bad = np.argwhere(~ok)
    assert bad.size == 0, (f"{len(bad)} FP8 keys out of tolerance, first at {bad[0]}: "
                           f"gpu {g[tuple(bad[0])]!r} oracle {t[tuple(bad[0])]!r}")
    return {"n": int(g.size), "within_1ulp": int((within & ~sat).sum()), "saturated": int(sat.sum())}


def compare_tokens_fp8(wl, gathered_k, gathered_v, entries, freqs, style: int, facts: FactCache,
                       k_scale: float, v_scale: float) -> dict:
    """As compare_tokens, for an E4M3 cache (gathered rows are uint8 bits)."""
    dtype = wl.spec.kv_dtype
    stats = {"n": 0, "within_1ulp": 0, "saturated": 0, "v_saturated": 0}
    for i, (f, j, p, _) in enumerate(entries):
        Kj, Vj = facts.token(f, j)
        want_v = oinject.e4m3_value(Vj, dtype, v_scale)
        assert np.array_equal(np.asarray(gathered_v[i]), want_v), f"FP8 V of fact {f} token {j} differs"
        stats["v_saturated"] += int((np.abs(numerics.e4m3_bits_to_f64(want_v)) == numerics.E4M3_MAX).sum())
        x = numerics.decode(Kj, dtype)
        o = oinject.rotated_key_rows(Kj, p, freqs, style, dtype)
        st = check_rotated_e4m3(gathered_k[i], o, x, style, k_scale)
        for key in ("n", "within_1ulp", "saturated"):
            stats[key] += st[key]
    return stats
