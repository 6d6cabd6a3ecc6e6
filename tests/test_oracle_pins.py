"""Pins of the fp64 oracle against things other than itself.

Each check ties an oracle function to a closed form, a hand-derived value, an
invariant, a textbook formulation or brute force (InferScale, Theorems 3 and 6;
RoFormer's rotation; the published Llama 3.1 RoPE scaling; the bf16 format;
vLLM's block-table slot mapping).  CPU only.
"""
import cmath
import itertools
import math
import os

import numpy as np
import pytest

from oracle import attention, inject, model, numerics, retrieval, rope

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


# ---------------------------------------------------------------- bf16 format

def test_bf16_rounding_golden():
    for row in _rows("bf16_rne.txt"):
        x = float(row[0])
        want = int(row[1], 16)
        got = int(numerics.f64_to_bf16_bits(np.array([x]))[0])
        assert got == want, (row, hex(got))


def test_bf16_rounding_matches_torch_on_fp32_inputs():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e-39,
                        rng.standard_normal(2000) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = numerics.f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_decode_roundtrip():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = numerics.bf16_bits_to_f64(bits)
    finite = np.isfinite(vals)
    back = numerics.f64_to_bf16_bits(vals[finite])
    # every finite bf16 re-encodes to itself
    assert np.array_equal(back, bits[finite])


def test_ulp_closed_forms():
    assert numerics.ulp(np.array([1.0]), "bf16")[0] == 2.0 ** -7
    assert numerics.ulp(np.array([1.99]), "bf16")[0] == 2.0 ** -7
    assert numerics.ulp(np.array([-2.0]), "bf16")[0] == 2.0 ** -6
    assert numerics.ulp(np.array([0.75]), "bf16")[0] == 2.0 ** -8
    assert numerics.ulp(np.array([1.0]), "f32")[0] == 2.0 ** -23
    assert numerics.ulp(np.array([0.0]), "bf16")[0] == 2.0 ** -133


# ---------------------------------------------------------------- FP8 E4M3 format

def test_e4m3_rounding_golden():
    for row in _rows("e4m3_rne_sat.txt"):
        x = float(row[0])
        want = int(row[1], 16)
        got = int(numerics.f64_to_e4m3_bits(np.array([x]))[0])
        assert got == want, (row, hex(got))


def test_e4m3_decode_roundtrip_all_codes():
    bits = np.arange(256, dtype=np.uint8)
    vals = numerics.e4m3_bits_to_f64(bits)
    nan = np.isnan(vals)
    assert np.array_equal(np.nonzero(nan)[0], [0x7F, 0xFF])
    assert np.array_equal(numerics.f64_to_e4m3_bits(vals[~nan]), bits[~nan])
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0) and pos[0] == 0.0 and pos[-1] == 448.0


def test_e4m3_matches_torch_float8_within_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * 4, rng.uniform(-448, 448, 5000),
                        rng.standard_normal(5000) * 2e-3]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = numerics.f64_to_e4m3_bits(x.astype(np.float64))
    assert np.array_equal(got, ref)
    dec = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    ours = numerics.e4m3_bits_to_f64(np.arange(256, dtype=np.uint8))
    fin = ~np.isnan(ours)
    assert np.array_equal(np.isnan(dec), ~fin) and np.array_equal(dec[fin].astype(np.float64), ours[fin])


def test_e4m3_ulp_closed_forms():
    assert numerics.ulp(np.array([1.0]), "e4m3")[0] == 2.0 ** -3
    assert numerics.ulp(np.array([448.0]), "e4m3")[0] == 32.0
    assert numerics.ulp(np.array([2.0 ** -7]), "e4m3")[0] == 2.0 ** -9
    assert numerics.ulp(np.array([0.0]), "e4m3")[0] == 2.0 ** -9


def test_inject_fp8_cache_quantises_scaled_values():
    """E4M3 cache: K is the rotated key times fp32(1 / k_scale) rounded once;
    V is fp32(v) * fp32(1 / v_scale) rounded; untouched rows keep the canary."""
    rng = np.random.default_rng(11)
    L, H, D, bs, NB = 2, 2, 8, 4, 6
    lengths = np.array([3, 4])
    store = {f: (numerics.encode(rng.standard_normal((lengths[f], L, H, D)) * 3, "bf16"),
                 numerics.encode(rng.standard_normal((lengths[f], L, H, D)) * 3, "bf16")) for f in range(2)}
    cache = np.full((L, 2, NB, bs, H, D), 0x7F, dtype=np.uint8)
    before = cache.copy()
    row = [2, 5, 0, 1, 3, 4]
    w = rope.inv_freq(D, 1e4)
    ks, vs = 0.37, 0.011                     # the V scale drives values past 448: saturation
    plan, T, slots = inject.inject(cache, "bf16", lambda f: store[f], [1, 0], lengths, 5, row, bs, w, 0,
                                   cache_dtype="e4m3", k_scale=ks, v_scale=vs)
    touched = np.zeros(cache.shape, dtype=bool)
    saturated = 0
    for (f, j, p), s in zip(plan, slots):
        blk, off = divmod(int(s), bs)
        touched[:, :, blk, off] = True
        krot = rope.rotate(numerics.decode(store[f][0][j], "bf16"), p, w, 0)
        kq = numerics.e4m3_bits_to_f64(cache[:, 0, blk, off])
        rk, rv = np.float32(1 / np.float64(np.float32(ks))), np.float32(1 / np.float64(np.float32(vs)))
        # one rounding of k * r_k: within half an E4M3 ulp
        assert np.all(np.abs(kq - krot * float(rk)) <= 0.5 * numerics.ulp(kq, "e4m3") + 1e-12)
        v = numerics.decode(store[f][1][j], "bf16")
        vq = numerics.e4m3_bits_to_f64(cache[:, 1, blk, off])
        target = (v.astype(np.float32) * rv).astype(np.float64)
        sat = np.abs(target) > 448
        saturated += int(sat.sum())
        assert np.all(vq[sat] == np.sign(target[sat]) * 448.0)
        assert np.all(np.abs(vq - target)[~sat] <= 0.5 * numerics.ulp(vq, "e4m3")[~sat])
    assert saturated > 0
    assert np.array_equal(cache[~touched], before[~touched])


# ---------------------------------------------------------------- frequencies

def test_inv_freq_plain_closed_forms():
    w = rope.inv_freq(64, 1.0e4)
    assert w.shape == (32,)
    assert w[0] == 1.0
    for i, want in [(8, 1e-1), (16, 1e-2), (24, 1e-3)]:
        assert math.isclose(w[i], want, rel_tol=1e-14)
    assert np.all(np.diff(w) < 0)
    # geometric: consecutive ratio is theta^(-2/D)
    assert np.allclose(w[1:] / w[:-1], 1.0e4 ** (-2.0 / 64), rtol=1e-13)


def _llama3(D=128, theta=5.0e5):
    return rope.inv_freq(D, theta, scaling=1, factor=8.0, low_freq_factor=1.0,
                         high_freq_factor=4.0, original_max_pos=8192)


def test_llama31_scaling_regimes():
    base = rope.inv_freq(128, 5.0e5)
    sc = _llama3()
    lam = 2 * math.pi / base
    hi = lam < 8192 / 4.0
    lo = lam > 8192 / 1.0
    mid = ~hi & ~lo
    assert hi.sum() > 0 and lo.sum() > 0 and mid.sum() > 0
    assert np.array_equal(sc[hi], base[hi])                 # high frequencies untouched
    assert np.array_equal(sc[lo], base[lo] / 8.0)           # low frequencies exactly / factor
    assert np.all(sc[mid] < base[mid]) and np.all(sc[mid] > base[mid] / 8.0)
    assert np.all(np.diff(sc) < 0)                          # still strictly decreasing


def test_llama31_scaling_continuous_and_quadratic_in_band():
    # Evaluate the rule on a dense synthetic frequency grid through the band
    # edges: the scaled frequency is continuous at both edges, and inside the
    # band scaled/w is affine in w (it is 1/8 + (7/8) * s with s affine in w).
    L0 = 8192.0
    for w_edge, ratio in [(2 * math.pi / (L0 / 4.0), 1.0), (2 * math.pi / L0, 1.0 / 8.0)]:
        for eps in (1e-9, -1e-9):
            w = w_edge * (1 + eps)
            theta = w ** -2.0            # D = 4: inv_freq[1] = theta^(-1/2) = w
            got = rope.inv_freq(4, theta, 1, 8.0, 1.0, 4.0, int(L0))[1]
            assert math.isclose(got / w, ratio, rel_tol=1e-6)
    ws = np.linspace(2 * math.pi / (L0 / 4.0) * 0.99, 2 * math.pi / L0 * 1.01, 7)
    r = np.array([rope.inv_freq(4, w ** -2.0, 1, 8.0, 1.0, 4.0, int(L0))[1] / w for w in ws])
    second_diff = r[2:] - 2 * r[1:-1] + r[:-2]
    assert np.max(np.abs(second_diff)) < 1e-12
    assert np.all(np.diff(r) < 0) or np.all(np.diff(r) > 0)


# ---------------------------------------------------------------- rotation

def test_rotation_hand_value():
    # D = 2, theta arbitrary: inv_freq = [1]; rotating (1, 0) by p = 1 gives (cos 1, sin 1).
    w = rope.inv_freq(2, 1.0e4)
    assert w[0] == 1.0
    out = rope.rotate(np.array([1.0, 0.0]), 1, w, 0)
    assert np.allclose(out, [math.cos(1.0), math.sin(1.0)], atol=1e-15)
    out = rope.rotate(np.array([0.0, 1.0]), 1, w, 0)
    assert np.allclose(out, [-math.sin(1.0), math.cos(1.0)], atol=1e-15)


def test_rotation_pairing_styles():
    # D = 4: pair 0 uses frequency 1.  NeoX pairs (0, 2); interleaved pairs (0, 1).
    w = rope.inv_freq(4, 100.0)          # [1, 0.1]
    e0 = np.array([1.0, 0.0, 0.0, 0.0])
    neox = rope.rotate(e0, 2, w, 0)
    inter = rope.rotate(e0, 2, w, 1)
    assert np.allclose(neox, [math.cos(2), 0, math.sin(2), 0], atol=1e-15)
    assert np.allclose(inter, [math.cos(2), math.sin(2), 0, 0], atol=1e-15)
    e3 = np.array([0.0, 0.0, 0.0, 1.0])
    assert np.allclose(rope.rotate(e3, 2, w, 0), [0, -math.sin(0.2), 0, math.cos(0.2)], atol=1e-15)
    assert np.allclose(rope.rotate(e3, 2, w, 1), [0, 0, -math.sin(0.2), math.cos(0.2)], atol=1e-15)


@pytest.mark.parametrize("style", [0, 1])
def test_rotation_is_complex_multiplication(style):
    # RoFormer's formulation: pair (a, b) as a + ib multiplied by exp(i p w).
    rng = np.random.default_rng(1)
    D = 16
    w = rope.inv_freq(D, 1.0e4)
    x = rng.standard_normal(D)
    p = 12345
    ia, ib = (np.arange(8), np.arange(8) + 8) if style == 0 else (np.arange(0, 16, 2), np.arange(1, 16, 2))
    want = np.empty(D)
    for i in range(8):
        z = complex(x[ia[i]], x[ib[i]]) * cmath.exp(1j * p * w[i])
        want[ia[i]], want[ib[i]] = z.real, z.imag
    assert np.allclose(rope.rotate(x, p, w, style), want, atol=1e-12)


@pytest.mark.parametrize("style", [0, 1])
def test_rotation_group_properties(style):
    rng = np.random.default_rng(2)
    D = 32
    w = _llama3(D, 5.0e5)
    x = rng.standard_normal((5, D))
    assert np.array_equal(rope.rotate(x, 0, w, style), x)                       # R(0) = I
    for p in (1, 77, 4096, 30000):
        y = rope.rotate(x, p, w, style)
        assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    # R(n) R(m) = R(m + n)  and  R(-m) R(m) = I
    assert np.allclose(rope.rotate(rope.rotate(x, 300, w, style), 45, w, style),
                       rope.rotate(x, 345, w, style), atol=1e-12)
    assert np.allclose(rope.rotate(rope.rotate(x, 999, w, style), -999, w, style), x, atol=1e-12)


@pytest.mark.parametrize("style", [0, 1])
def test_theorem6_scores_depend_only_on_offset(style):
    # Theorem 6: <R(m) q, R(n) k> depends only on m - n, so keys re-rotated to
    # any position give the same attention scores as a prefill there.
    rng = np.random.default_rng(3)
    D = 64
    w = rope.inv_freq(D, 1.0e4)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    for m, n in [(10, 3), (500, 499), (7, 7), (3000, 10)]:
        ref = rope.rotate(q, m, w, style) @ rope.rotate(k, n, w, style)
        for c in (1, 64, 12345):
            got = rope.rotate(q, m + c, w, style) @ rope.rotate(k, n + c, w, style)
            assert math.isclose(got, ref, rel_tol=1e-9, abs_tol=1e-10)


# ---------------------------------------------------------------- retrieval

def test_cosine_closed_forms():
    X = np.array([[1.0, 1.0], [0.0, 3.0], [-2.0, 0.0], [5.0, 0.0], [0.0, 0.0]])
    s = retrieval.cosine_scores(np.array([2.0, 0.0]), X)
    assert np.allclose(s, [1 / math.sqrt(2), 0.0, -1.0, 1.0, 0.0], atol=1e-15)


def _brute_topk(scores, ids, k):
    # An entry is selected iff fewer than k entries beat it (higher score, or
    # equal score and lower id); its rank is the number that beat it.
    out = []
    for a in range(len(ids)):
        beat = sum(1 for b in range(len(ids))
                   if scores[b] > scores[a] or (scores[b] == scores[a] and ids[b] < ids[a]))
        if beat < k:
            out.append((beat, ids[a], scores[a]))
    out.sort()
    return [o[1] for o in out], [o[2] for o in out]


def test_topk_brute_force_tiny_stores_with_ties():
    rng = np.random.default_rng(4)
    for trial in range(300):
        n = int(rng.integers(1, 12))
        scores = rng.integers(-3, 4, size=n).astype(np.float64) / 4.0   # many ties
        ids = rng.permutation(100)[:n].astype(np.int64)
        k = int(rng.integers(1, 14))
        want_ids, want_sc = _brute_topk(scores, ids, k)
        got_ids, got_sc = retrieval.topk(scores, ids, k)
        assert list(got_ids) == want_ids
        assert list(got_sc) == want_sc


def test_topk_exhaustive_subset_maximises_score_sum():
    rng = np.random.default_rng(5)
    for _ in range(50):
        n, k = 8, 3
        s = rng.standard_normal(n)
        ids = np.arange(n)
        best = max(itertools.combinations(range(n), k), key=lambda c: sum(s[list(c)]))
        got, _ = retrieval.topk(s, ids, k)
        assert sorted(got) == sorted(best)


def test_planted_query_ranks_its_fact_first():
    rng = np.random.default_rng(6)
    X = rng.standard_normal((64, 64))
    X /= np.linalg.norm(X, axis=1, keepdims=True)
    ids = np.arange(1000, 1064)
    got, sc = retrieval.retrieve(X[17], X, ids, 4)
    assert got[0] == 1017 and math.isclose(sc[0], 1.0, rel_tol=1e-14)
    assert np.all(np.diff(sc) <= 0)


# ---------------------------------------------------------------- slot mapping / composition

def test_slot_mapping_golden():
    for row in _rows("slot_mapping.txt"):
        bs, table, p, want = int(row[0]), [int(t) for t in row[1].split(",")], int(row[2]), int(row[3])
        assert inject.slot(p, table, bs) == want


def test_compose_positions_and_lengths():
    lengths = np.array([3, 1, 4, 2])
    plan, T = inject.compose([2, 0, 3], lengths, 10)
    assert T == 4 + 3 + 2 == len(plan)
    assert [p for _, _, p in plan] == list(range(10, 19))
    assert [(f, j) for f, j, _ in plan] == [(2, 0), (2, 1), (2, 2), (2, 3), (0, 0), (0, 1), (0, 2),
                                            (3, 0), (3, 1)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_inject_tiny_canaries_and_copies(dtype):
    rng = np.random.default_rng(7)
    L, H, D, bs, NB = 2, 2, 8, 4, 6
    lengths = np.array([3, 5, 2])
    store = {}
    for f in range(3):
        K = rng.standard_normal((lengths[f], L, H, D))
        V = rng.standard_normal((lengths[f], L, H, D))
        store[f] = (numerics.encode(K, dtype), numerics.encode(V, dtype))
    canary = 0x7FA5 if dtype == "bf16" else np.float32(np.nan)
    cache = np.full((L, 2, NB, bs, H, D), canary, dtype=np.uint16 if dtype == "bf16" else np.float32)
    before = cache.copy()
    row = [5, 0, 3, 1, 2, 4]
    w = rope.inv_freq(D, 1e4)
    plan, T, slots = inject.inject(cache, dtype, lambda f: store[f], [1, 2], lengths, 6, row, bs, w, 0)
    assert T == 7 and list(slots) == [inject.slot(p, row, bs) for p in range(6, 13)]
    touched = np.zeros(cache.shape, dtype=bool)
    for (f, j, p), s in zip(plan, slots):
        blk, off = divmod(int(s), bs)
        touched[:, :, blk, off] = True
        assert np.array_equal(cache[:, 1, blk, off], store[f][1][j])        # V bit-exact
        krot = rope.rotate(numerics.decode(store[f][0][j], dtype), p, w, 0)
        assert np.array_equal(cache[:, 0, blk, off], numerics.encode(krot, dtype))
    same = (cache.view(np.uint8) == before.view(np.uint8)).reshape(cache.shape + (-1,)).all(-1)
    assert same[~touched].all()


# ---------------------------------------------------------------- attention, RMSNorm, SiLU by hand

def test_causal_attention_hand_weights():
    """Softmax attention (Vaswani et al., scaled dot product) worked by hand.

    D = 2, one head.  q = (sqrt(2)·ln 2, 0) and k_s = (s, 0), so after the
    1/sqrt(D) scale the logit of key s is s·ln 2 and its softmax weight is
    proportional to 2^s: a query that sees keys 0, 1, 2 weighs them 1/7, 2/7,
    4/7.  Keys sit at positions 5, 7, 9 and queries at 5, 8, 9, so the causal
    mask has to compare positions (key position <= query position), not
    indices: the query at 8 sees keys 0 and 1 only (weights 1/3, 2/3)."""
    a = math.sqrt(2.0) * math.log(2.0)
    q = np.array([[a, 0.0], [a, 0.0], [a, 0.0]])[:, None, :]
    k = np.array([[0.0, 0.0], [1.0, 0.0], [2.0, 0.0]])[:, None, :]
    v = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])[:, None, :]
    out = attention.causal_attention(q, np.array([5, 8, 9]), k, np.array([5, 7, 9]), v)
    want = np.array([[1.0, 0.0], [1 / 3, 2 / 3], [5 / 7, 6 / 7]])
    assert np.max(np.abs(out[:, 0, :] - want)) < 1e-15


def test_causal_attention_grouped_query_heads():
    """Grouped-query attention: with 4 query heads over 2 KV heads, query heads
    0 and 1 read KV head 0 and heads 2 and 3 read KV head 1.  Every key gets the
    same logit (zero query), so each output is the plain mean of the visible
    values of its KV head."""
    q = np.zeros((2, 4, 2))
    k = np.ones((2, 2, 2))
    v = np.array([[[1.0, 2.0], [10.0, 20.0]],
                  [[3.0, 4.0], [30.0, 40.0]]])                  # [token][kv head][D]
    out = attention.causal_attention(q, np.array([0, 1]), k, np.array([0, 1]), v)
    for h in range(4):
        g = h // 2
        assert np.array_equal(out[0, h], v[0, g])
        assert np.max(np.abs(out[1, h] - (v[0, g] + v[1, g]) / 2)) < 1e-15


def test_rmsnorm_hand_values():
    """RMSNorm without gain (Zhang and Sennrich): x / sqrt(mean(x²) + eps).
    (3, 4): mean square 12.5, so the result is (3, 4)/sqrt(12.5); a constant
    vector c·1 maps to 1 (up to eps); the scale of x does not matter."""
    y = model.rmsnorm(np.array([3.0, 4.0]), eps=0.0)
    assert np.max(np.abs(y - np.array([3.0, 4.0]) / math.sqrt(12.5))) < 1e-15
    assert abs(y[0] - 0.848528137423857) < 1e-14 and abs(y[1] - 1.131370849898476) < 1e-14
    assert np.max(np.abs(model.rmsnorm(np.full(7, -2.5), eps=0.0) + 1.0)) < 1e-15
    x = np.random.default_rng(3).standard_normal((4, 9))
    assert np.max(np.abs(model.rmsnorm(x * 1e3, eps=0.0) - model.rmsnorm(x, eps=0.0))) < 1e-13
    # eps sits under the square root: (3, 4) with eps = 12.5 halves the mean square's root.
    y = model.rmsnorm(np.array([3.0, 4.0]), eps=12.5)
    assert np.max(np.abs(y - np.array([3.0, 4.0]) / 5.0)) < 1e-15


def test_silu_hand_values():
    """SiLU(x) = x·sigmoid(x) (Elfwing et al.; Hendrycks and Gimpel).
    SiLU(0) = 0; SiLU(ln 3) = ln 3 · 3/4; SiLU(-ln 3) = -ln 3 · 1/4;
    SiLU(x) -> x as x -> +inf and -> 0 as x -> -inf."""
    ln3 = math.log(3.0)
    y = model.silu(np.array([0.0, ln3, -ln3, 40.0, -40.0]))
    assert y[0] == 0.0
    assert abs(y[1] - 0.75 * ln3) < 1e-15 and abs(y[2] + 0.25 * ln3) < 1e-15
    assert abs(y[3] - 40.0) < 1e-12 and abs(y[4]) < 1e-14


# ---------------------------------------------------------------- Theorem 3 / 6 on tiny attention

def _tiny_model(rng, dm=16, Hq=4, Hk=2, D=8):
    s = 1 / math.sqrt(dm)
    return (rng.standard_normal((dm, Hq * D)) * s, rng.standard_normal((dm, Hk * D)) * s,
            rng.standard_normal((dm, Hk * D)) * s, Hq, Hk, D)


@pytest.mark.parametrize("style,scaled", [(0, False), (1, False), (0, True)])
def test_theorem3_injection_equals_prompt_prefill(style, scaled):
    rng = np.random.default_rng(8 + style + 2 * scaled)
    Wq, Wk, Wv, Hq, Hk, D = _tiny_model(rng)
    freqs = (rope.inv_freq(D, 5e5, 1, 8.0, 1.0, 4.0, 16) if scaled else rope.inv_freq(D, 1e4))
    dm = Wq.shape[0]
    start, lengths = 5, np.array([3, 2, 4])
    x_prefix = rng.standard_normal((start, dm))
    x_fact = [rng.standard_normal((int(n), dm)) for n in lengths]
    x_query = rng.standard_normal((3, dm))
    order = [2, 0, 1]

    # Prompt injection: prefill [prefix | facts in order | query] at positions 0..T-1.
    x_all = np.concatenate([x_prefix] + [x_fact[f] for f in order] + [x_query])
    T = x_all.shape[0]
    out_prompt = attention.prefill(x_all, np.arange(T), Wq, Wk, Wv, Hq, Hk, freqs, style)[0]

    # KV injection through the paged cache.
    bs, NB = 4, 8
    row = list(rng.permutation(NB))
    cache = np.zeros((1, 2, NB, bs, Hk, D))
    _, _, k_rot, _, v = attention.prefill(x_prefix, np.arange(start), Wq, Wk, Wv, Hq, Hk, freqs, style)
    for p in range(start):
        blk, off = divmod(inject.slot(p, row, bs), bs)
        cache[0, 0, blk, off], cache[0, 1, blk, off] = k_rot[p], v[p]

    def fact_kv(f):   # encoded once, alone, before RoPE: [len][L=1][Hk][D]
        return attention.heads(x_fact[f], Wk, Hk)[:, None], attention.heads(x_fact[f], Wv, Hk)[:, None]

    _, seg_len, _ = inject.inject(cache, "f64", fact_kv, order, lengths, start, row, bs, freqs, style)
    assert seg_len == lengths.sum()
    qpos = np.arange(start + seg_len, T)
    q = attention.heads(x_query, Wq, Hq)
    q_rot = rope.rotate(q, qpos[:, None], freqs, style)
    kq = rope.rotate(attention.heads(x_query, Wk, Hk), qpos[:, None], freqs, style)
    vq = attention.heads(x_query, Wv, Hk)
    for i, p in enumerate(qpos):
        blk, off = divmod(inject.slot(int(p), row, bs), bs)
        cache[0, 0, blk, off], cache[0, 1, blk, off] = kq[i], vq[i]
    K, V = attention.read_paged(cache, row, bs, T)
    out_inject = attention.causal_attention(q_rot, qpos, K, np.arange(T), V)
    assert np.max(np.abs(out_inject - out_prompt[qpos])) < 1e-12


def test_theorem6_stored_key_rerotated_equals_key_computed_in_place():
    rng = np.random.default_rng(11)
    Wq, Wk, Wv, Hq, Hk, D = _tiny_model(rng)
    freqs = rope.inv_freq(D, 1e4)
    x = rng.standard_normal((6, Wq.shape[0]))
    # Encode the fact alone at positions 0..5 and keep its keys before RoPE.
    _, _, _, k_pre, _ = attention.prefill(x, np.arange(6), Wq, Wk, Wv, Hq, Hk, freqs, 0)
    for start in (0, 17, 4093):
        pos = np.arange(start, start + 6)
        _, _, k_at, _, _ = attention.prefill(x, pos, Wq, Wk, Wv, Hq, Hk, freqs, 0)
        rerot = np.stack([inject.rotated_key_rows(k_pre[t][None], int(pos[t]), freqs, 0, "f64")[0]
                          for t in range(6)])
        assert np.max(np.abs(rerot - k_at)) < 1e-12
