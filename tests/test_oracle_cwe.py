"""Pins of the Context-Window Encoding oracle (``oracle/cwe.py``) and of the
tiny decoder that produces the encodings (``oracle/model.py``).

What the pages fix, checked independently of the oracle's own formulas:
* w = 0 is independent encoding, and only the fact's tokens are kept;
* in a one-layer model a token's K/V depend on that token alone, so the
  window cannot change them (cross-fact context reaches K/V only through the
  layers below);
* stored keys are taken before RoPE, and attention depends only on relative
  positions (Theorem 6), so the stored K/V do not depend on where the
  encoded sequence starts;
* with the whole conversation as the window, the captured K/V equal those of
  the joint prefill of the conversation, and injecting them (with the turns
  before) reproduces the joint prefill of a following query exactly
  (Theorem 3 with KV encoded in the joint context);
* with a shorter window the deeper layers' K/V differ (the approximation the
  pages measure).
Mutations of the oracle are planted at the end; each must fail a pin.
"""
import numpy as np
import pytest

from oracle import cwe, model, rope


def _setup(n_layers=3, seed=0, n_turns=9, d=32, style=0):
    rng = np.random.default_rng(seed)
    m = model.make_model(rng, n_layers, d, 4, 2, 16, 64, theta=1.0e4, style=style)
    turns = [rng.standard_normal((int(n), d)) for n in rng.integers(2, 7, size=n_turns)]
    return m, turns, rng


def _independent(m, turns, i):
    _, kv = model.forward(m, turns[i], np.arange(len(turns[i])))
    return np.stack([k for k, _ in kv], 1), np.stack([v for _, v in kv], 1)


def test_zero_window_is_independent_encoding():
    m, turns, _ = _setup()
    for i in (0, 4, 8):
        K, V = cwe.cwe_fact_kv(m, turns, i, 0)
        Ki, Vi = _independent(m, turns, i)
        assert np.array_equal(K, Ki) and np.array_equal(V, Vi)
        assert K.shape == (len(turns[i]), 3, 2, 16)


def test_one_layer_kv_do_not_depend_on_the_window():
    m, turns, _ = _setup(n_layers=1)
    for w in (1, 3, 8):
        K, V = cwe.cwe_fact_kv(m, turns, 6, w)
        Ki, Vi = _independent(m, turns, 6)
        assert np.allclose(K, Ki, rtol=0, atol=1e-13) and np.allclose(V, Vi, rtol=0, atol=1e-13)


@pytest.mark.parametrize("style", [0, 1])
def test_stored_kv_do_not_depend_on_the_start_position(style):
    m, turns, _ = _setup(style=style)
    for offset in (1, 37, 4096 + 13):
        K0, V0 = cwe.cwe_fact_kv(m, turns, 5, 3, offset=0)
        K1, V1 = cwe.cwe_fact_kv(m, turns, 5, 3, offset=offset)
        assert np.max(np.abs(K0 - K1)) < 1e-10 and np.max(np.abs(V0 - V1)) < 1e-10


def test_full_window_equals_the_joint_prefill_of_the_conversation():
    m, turns, _ = _setup()
    x = np.concatenate(turns)
    _, kv = model.forward(m, x, np.arange(len(x)))
    start = np.cumsum([0] + [len(t) for t in turns])
    for i in (0, 3, 8):
        K, V = cwe.cwe_fact_kv(m, turns, i, w=i)
        for l, (k, v) in enumerate(kv):
            assert np.max(np.abs(K[:, l] - k[start[i]:start[i + 1]])) < 1e-12
            assert np.max(np.abs(V[:, l] - v[start[i]:start[i + 1]])) < 1e-12


def test_shorter_window_changes_only_the_deeper_layers():
    m, turns, _ = _setup()
    K, V = cwe.cwe_fact_kv(m, turns, 7, w=2)
    Ki, Vi = _independent(m, turns, 7)
    assert np.max(np.abs(K[:, 0] - Ki[:, 0])) < 1e-12          # layer 0 is token-local
    assert np.max(np.abs(K[:, 1:] - Ki[:, 1:])) > 1e-3          # deeper layers see the window
    assert np.max(np.abs(V[:, 1:] - Vi[:, 1:])) > 1e-3


def _inject_and_query(m, fact_kv_rows, positions, q_tokens, q_pos):
    """Serving: facts' K/V in the cache (rotated at their positions), then the
    query prefilled through every layer on top of them."""
    past = []
    for l in range(len(m.layers)):
        k = np.concatenate([K[:, l] for K, _ in fact_kv_rows])
        v = np.concatenate([V[:, l] for _, V in fact_kv_rows])
        past.append((rope.rotate(k, positions[:, None], m.freqs, m.style), positions, v))
    h, _ = model.forward(m, q_tokens, q_pos, past=past)
    return h


def test_injected_joint_context_kv_reproduce_the_joint_prefill():
    """Theorem 3 beyond one layer: with KV encoded in the joint context, every
    turn captured with its whole history, injection equals prompt prefill."""
    m, turns, rng = _setup()
    q = rng.standard_normal((4, 32))
    x = np.concatenate(turns + [q])
    h_joint, _ = model.forward(m, x, np.arange(len(x)))
    n_ctx = sum(len(t) for t in turns)
    rows = [cwe.cwe_fact_kv(m, turns, i, w=i) for i in range(len(turns))]
    h_inj = _inject_and_query(m, rows, np.arange(n_ctx), q, np.arange(n_ctx, n_ctx + 4))
    assert np.max(np.abs(h_inj - h_joint[n_ctx:])) < 1e-10
    # independent encoding of the same turns does not reproduce it
    rows0 = [cwe.cwe_fact_kv(m, turns, i, w=0) for i in range(len(turns))]
    h0 = _inject_and_query(m, rows0, np.arange(n_ctx), q, np.arange(n_ctx, n_ctx + 4))
    assert np.max(np.abs(h0 - h_joint[n_ctx:])) > 1e-3


# ---------------------------------------------------------------- planted mistakes

def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def test_mutation_capture_keeps_the_window_tokens(monkeypatch):
    def first_tokens(kv, window_len):          # as many tokens as the fact, from the front
        n = len(kv[0][0]) - window_len
        return (np.stack([k[:n] for k, _ in kv], axis=1), np.stack([v[:n] for _, v in kv], axis=1))
    monkeypatch.setattr(cwe, "capture", first_tokens)
    assert _fails(test_full_window_equals_the_joint_prefill_of_the_conversation)


def test_mutation_window_of_following_turns(monkeypatch):
    monkeypatch.setattr(cwe, "window_turns", lambda i, w: range(i + 1, i + 1 + w))
    def run():
        m, turns, _ = _setup()
        turns = turns + [turns[0]] * 9                     # room for "following" turns
        K, _ = cwe.cwe_fact_kv(m, turns, 3, w=3)
        x = np.concatenate(turns[:4])
        _, kv = model.forward(m, x, np.arange(len(x)))
        s = sum(len(t) for t in turns[:3])
        assert np.max(np.abs(K[:, 2] - kv[2][0][s:])) < 1e-12
    assert _fails(run)


def test_mutation_keys_captured_after_rope(monkeypatch):
    orig = model.forward

    def post_rope(m, x, positions, past=None):
        h, kv = orig(m, x, positions, past)
        pos = np.asarray(positions)
        return h, [(rope.rotate(k, pos[:, None], m.freqs, m.style), v) for k, v in kv]
    monkeypatch.setattr(model, "forward", post_rope)
    assert _fails(test_stored_kv_do_not_depend_on_the_start_position, 0)


def test_mutation_window_ignored(monkeypatch):
    orig = cwe.encode_with_window
    monkeypatch.setattr(cwe, "encode_with_window", lambda m, turns, i, w, offset=0: orig(m, turns, i, 0, offset))
    assert _fails(test_full_window_equals_the_joint_prefill_of_the_conversation)
    assert _fails(test_shorter_window_changes_only_the_deeper_layers)
