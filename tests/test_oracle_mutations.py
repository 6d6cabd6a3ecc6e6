"""Plant plausible mistakes in the oracle (on the CPU) and check a pin catches each.

A pin set that a dropped term, a wrong sign, a wrong index or a swapped operand
slips through would not pin anything; each case below patches one oracle
function and requires at least one of the named pins to fail.
"""
import numpy as np
import pytest

import tests.test_oracle_pins as pins
from oracle import attention, inject, model, numerics, retrieval, rope


def _fails(fn, *args):
    try:
        fn(*args)
    except (AssertionError, IndexError, ValueError):
        return True
    return False


def _rotate_wrong_sign(x, position, freqs, style):
    x = np.asarray(x, dtype=np.float64)
    ia, ib = rope.pair_indices(x.shape[-1], style)
    phi = np.asarray(position, dtype=np.float64)[..., None] * freqs
    c, s = np.cos(phi), np.sin(phi)
    out = np.empty(np.broadcast_shapes(x.shape, phi.shape[:-1] + (x.shape[-1],)))
    out[..., ia] = x[..., ia] * c + x[..., ib] * s
    out[..., ib] = x[..., ib] * c - x[..., ia] * s
    return out


def _rotate_dropped_term(x, position, freqs, style):
    x = np.asarray(x, dtype=np.float64)
    ia, ib = rope.pair_indices(x.shape[-1], style)
    phi = np.asarray(position, dtype=np.float64)[..., None] * freqs
    out = np.empty(np.broadcast_shapes(x.shape, phi.shape[:-1] + (x.shape[-1],)))
    out[..., ia] = x[..., ia] * np.cos(phi) - x[..., ib] * np.sin(phi)
    out[..., ib] = x[..., ib] * np.cos(phi)
    return out


def _pairs_swapped(D, style):
    half = D // 2
    i = np.arange(half)
    return (2 * i, 2 * i + 1) if style == 0 else (i, i + half)


def test_mutation_rotation_sign(monkeypatch):
    monkeypatch.setattr(rope, "rotate", _rotate_wrong_sign)
    assert _fails(pins.test_rotation_hand_value)
    assert _fails(pins.test_rotation_is_complex_multiplication, 0)


def test_mutation_rotation_dropped_term(monkeypatch):
    monkeypatch.setattr(rope, "rotate", _rotate_dropped_term)
    assert _fails(pins.test_rotation_hand_value)
    assert _fails(pins.test_rotation_group_properties, 0)
    assert _fails(pins.test_theorem6_scores_depend_only_on_offset, 0)


def test_mutation_pairing_swapped(monkeypatch):
    monkeypatch.setattr(rope, "pair_indices", _pairs_swapped)
    assert _fails(pins.test_rotation_pairing_styles)


def test_mutation_frequency_exponent(monkeypatch):
    orig = rope.inv_freq

    def wrong(head_dim, theta, *a, **k):
        return orig(2 * head_dim, theta, *a, **k)[: head_dim // 2]      # theta^(-i/D)
    monkeypatch.setattr(rope, "inv_freq", wrong)
    assert _fails(pins.test_inv_freq_plain_closed_forms)


def test_mutation_llama3_factor_multiplied(monkeypatch):
    orig = rope.inv_freq

    def wrong(head_dim, theta, scaling=0, factor=1.0, *a, **k):
        return orig(head_dim, theta, scaling, 1.0 / factor, *a, **k)
    monkeypatch.setattr(rope, "inv_freq", wrong)
    assert _fails(pins.test_llama31_scaling_regimes)


def test_mutation_llama3_blend_swapped(monkeypatch):
    orig = rope.inv_freq

    def wrong(head_dim, theta, scaling=0, factor=1.0, low_freq_factor=1.0,
              high_freq_factor=1.0, original_max_pos=0):
        return orig(head_dim, theta, scaling, factor, high_freq_factor, low_freq_factor,
                    original_max_pos)                                      # low/high swapped
    monkeypatch.setattr(rope, "inv_freq", wrong)
    assert _fails(pins.test_llama31_scaling_regimes)


def test_mutation_slot_index_swapped(monkeypatch):
    monkeypatch.setattr(inject, "slot",
                        lambda p, row, bs: int(row[p % bs]) * bs + p // bs)
    assert _fails(pins.test_slot_mapping_golden)
    assert _fails(pins.test_theorem3_injection_equals_prompt_prefill, 0, False)


def test_mutation_position_off_by_one(monkeypatch):
    orig = inject.compose

    def wrong(fact_ids, lengths, start):
        return orig(fact_ids, lengths, start + 1)
    monkeypatch.setattr(inject, "compose", wrong)
    assert _fails(pins.test_theorem3_injection_equals_prompt_prefill, 0, False)
    assert _fails(pins.test_compose_positions_and_lengths)


def test_mutation_topk_ties_to_higher_id(monkeypatch):
    def wrong(scores, ids, k):
        order = np.lexsort((-np.asarray(ids), -np.asarray(scores, dtype=np.float64)))[:k]
        return np.asarray(ids)[order], np.asarray(scores, dtype=np.float64)[order]
    monkeypatch.setattr(retrieval, "topk", wrong)
    assert _fails(pins.test_topk_brute_force_tiny_stores_with_ties)


def test_mutation_cosine_unnormalised_query(monkeypatch):
    def wrong(q, X):
        X = np.asarray(X, dtype=np.float64)
        n = np.linalg.norm(X, axis=1)
        return np.where(n > 0, (X @ np.asarray(q, dtype=np.float64)) / np.where(n > 0, n, 1), 0.0)
    monkeypatch.setattr(retrieval, "cosine_scores", wrong)
    assert _fails(pins.test_cosine_closed_forms)


def test_mutation_bf16_double_rounding(monkeypatch):
    def wrong(x):
        f = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
        return ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)
    monkeypatch.setattr(numerics, "f64_to_bf16_bits", wrong)
    assert _fails(pins.test_bf16_rounding_golden)


def test_mutation_bf16_truncation(monkeypatch):
    def wrong(x):
        return (np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    monkeypatch.setattr(numerics, "f64_to_bf16_bits", wrong)
    assert _fails(pins.test_bf16_rounding_golden)


@pytest.mark.parametrize("which", ["k", "v"])
def test_mutation_scatter_drops_rotation_or_copy(monkeypatch, which):
    orig = inject.rotated_key_rows
    if which == "k":
        monkeypatch.setattr(inject, "rotated_key_rows",
                            lambda k, p, f, s, d: orig(k, 0, f, s, d))   # rotation skipped
        assert _fails(pins.test_theorem3_injection_equals_prompt_prefill, 0, False)
    else:
        orig_inject = inject.inject

        def wrong(cache, dt, fact_kv, *a):
            return orig_inject(cache, dt, lambda f: (fact_kv(f)[0], fact_kv(f)[0]), *a)  # V := K
        monkeypatch.setattr(inject, "inject", wrong)
        assert _fails(pins.test_inject_tiny_canaries_and_copies, "f32")
        assert _fails(pins.test_theorem3_injection_equals_prompt_prefill, 0, False)


def test_mutation_e4m3_ties_away_from_zero(monkeypatch):
    orig = numerics.f64_to_e4m3_bits

    def wrong(x):
        # nudge every exact tie upwards in magnitude before the correct rounding
        x = np.asarray(x, dtype=np.float64)
        return orig(x * (1 + 2.0 ** -40))
    monkeypatch.setattr(numerics, "f64_to_e4m3_bits", wrong)
    assert _fails(pins.test_e4m3_rounding_golden)


def test_mutation_e4m3_without_saturation(monkeypatch):
    orig = numerics.f64_to_e4m3_bits

    def wrong(x):
        x = np.asarray(x, dtype=np.float64)
        return np.where(np.abs(x) > 464, np.uint8(0x7F), orig(x)).astype(np.uint8)   # overflow -> NaN
    monkeypatch.setattr(numerics, "f64_to_e4m3_bits", wrong)
    assert _fails(pins.test_e4m3_rounding_golden)
    assert _fails(pins.test_inject_fp8_cache_quantises_scaled_values)


def test_mutation_e4m3_exponent_bias(monkeypatch):
    orig = numerics.e4m3_bits_to_f64
    monkeypatch.setattr(numerics, "e4m3_bits_to_f64", lambda b: orig(b) * 2.0)      # bias 6 for 7
    assert _fails(pins.test_e4m3_decode_roundtrip_all_codes)


def test_mutation_fp8_value_scale_multiplied(monkeypatch):
    orig = inject.e4m3_value
    monkeypatch.setattr(inject, "e4m3_value", lambda v, dt, s: orig(v, dt, 1.0 / s))
    assert _fails(pins.test_inject_fp8_cache_quantises_scaled_values)


def _attention_variant(mask, scale, weights, head_of):
    """causal_attention with one step replaced: the mask test, the logit scale,
    the softmax weights or the query-head -> KV-head map."""
    def fn(q_rot, q_pos, k_rot, k_pos, v):
        Tq, Hq, D = q_rot.shape
        Hk = k_rot.shape[1]
        out = np.zeros((Tq, Hq, D))
        for i in range(Tq):
            visible = mask(np.asarray(k_pos), q_pos[i])
            for h in range(Hq):
                g = head_of(h, Hq, Hk)
                logits = k_rot[visible, g, :] @ q_rot[i, h, :] * scale(D)
                w = weights(logits)
                out[i, h] = w @ v[visible, g, :]
        return out
    return fn


def _softmax(z):
    w = np.exp(z - z.max())
    return w / w.sum()


_MASK = lambda kp, qp: kp <= qp                                      # noqa: E731
_SCALE = lambda D: 1.0 / np.sqrt(D)                                  # noqa: E731
_HEAD = lambda h, Hq, Hk: h // (Hq // Hk)                            # noqa: E731


@pytest.mark.parametrize("mistake", ["strict_mask", "index_mask", "no_scale", "uniform", "head_mod"])
def test_mutation_causal_attention(monkeypatch, mistake):
    mask, scale, weights, head_of = _MASK, _SCALE, _softmax, _HEAD
    if mistake == "strict_mask":
        mask = lambda kp, qp: kp < qp                                 # noqa: E731
    elif mistake == "index_mask":                                     # key index read as its position
        mask = lambda kp, qp: np.arange(len(kp)) <= qp                # noqa: E731
    elif mistake == "no_scale":
        scale = lambda D: 1.0                                         # noqa: E731
    elif mistake == "uniform":
        weights = lambda z: np.full(z.shape, 1.0 / z.size)           # noqa: E731
    else:
        head_of = lambda h, Hq, Hk: h % Hk                            # noqa: E731
    monkeypatch.setattr(attention, "causal_attention", _attention_variant(mask, scale, weights, head_of))
    assert (_fails(pins.test_causal_attention_hand_weights)
            or _fails(pins.test_causal_attention_grouped_query_heads))


def test_mutation_causal_attention_unmutated_passes(monkeypatch):
    """The variant builder with no mistake passes both pins (so the cases above
    fail because of their one change)."""
    monkeypatch.setattr(attention, "causal_attention", _attention_variant(_MASK, _SCALE, _softmax, _HEAD))
    assert not _fails(pins.test_causal_attention_hand_weights)
    assert not _fails(pins.test_causal_attention_grouped_query_heads)


@pytest.mark.parametrize("mistake", ["sum", "eps_outside", "no_sqrt"])
def test_mutation_rmsnorm(monkeypatch, mistake):
    def wrong(x, eps=1e-6):
        x = np.asarray(x, dtype=np.float64)
        ms = np.mean(x * x, axis=-1, keepdims=True)
        if mistake == "sum":
            return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
        if mistake == "eps_outside":
            return x / (np.sqrt(ms) + eps)
        return x / (ms + eps)
    monkeypatch.setattr(model, "rmsnorm", wrong)
    assert _fails(pins.test_rmsnorm_hand_values)


@pytest.mark.parametrize("mistake", ["negated", "no_x"])
def test_mutation_silu(monkeypatch, mistake):
    if mistake == "negated":
        wrong = lambda x: x / (1.0 + np.exp(x))                       # noqa: E731  x·sigmoid(-x)
    else:
        wrong = lambda x: 1.0 / (1.0 + np.exp(-x))                    # noqa: E731  sigmoid alone
    monkeypatch.setattr(model, "silu", wrong)
    assert _fails(pins.test_silu_hand_values)
