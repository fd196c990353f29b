"""Pins of the oracle's input prologue (``oracle.forms.prologue``, [DP] §2.2
and the [DR] §3 layer design), CPU only: identities of SiLU and the sigmoid,
the limits where the answer is known in closed form, the unit norm and sign
of the keys, and planted mistakes that these pins must catch."""
import numpy as np
import pytest

from oracle import forms


def test_silu_odd_part_is_the_identity():
    # sigmoid(x) + sigmoid(-x) = 1, so x sigmoid(x) - (-x) sigmoid(-x) = x
    x = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(forms.silu(x) - forms.silu(-x), x, rtol=0, atol=1e-13)


def test_silu_limits():
    assert forms.silu(0.0) == 0.0
    h = np.array([1e-6, 1e-8])
    np.testing.assert_allclose(forms.silu(h) / h, 0.5, rtol=1e-6)   # slope sigmoid(0) at 0
    np.testing.assert_allclose(forms.silu(50.0), 50.0, rtol=1e-15)  # -> x for large x
    assert 0.0 > forms.silu(-50.0) > -1e-19                          # -> 0 from below


def test_keys_have_unit_norm_and_keep_signs():
    rng = np.random.default_rng(5)
    raw = rng.standard_normal((7, 3, 64)) * 2.0
    q, k, _ = forms.prologue(raw, raw[::-1], np.zeros(3))
    for x, r in ((q, raw), (k, raw[::-1])):
        np.testing.assert_allclose(np.linalg.norm(x, axis=-1), 1.0, rtol=0, atol=1e-14)
        assert np.array_equal(np.sign(x), np.sign(r))  # SiLU keeps the sign


def test_large_positive_inputs_reduce_to_plain_l2_normalisation():
    # SiLU is the identity to double precision above ~40
    rng = np.random.default_rng(6)
    raw = rng.uniform(40, 80, (5, 32))
    _, k, _ = forms.prologue(raw, raw, np.zeros(5))
    np.testing.assert_allclose(k, raw / np.linalg.norm(raw, axis=-1, keepdims=True), rtol=1e-14)


def test_zero_vector_maps_to_zero():
    raw = np.zeros((2, 16))
    raw[1, 3] = 1.0
    _, k, _ = forms.prologue(raw, raw, np.zeros(2))
    assert np.all(k[0] == 0.0)
    np.testing.assert_allclose(k[1], np.eye(16)[3])


def test_beta_maps():
    x = np.linspace(-20, 20, 81)
    _, _, b1 = forms.prologue(np.ones((1, 4)), np.ones((1, 4)), x, "sigmoid")
    _, _, b2 = forms.prologue(np.ones((1, 4)), np.ones((1, 4)), x, "2sigmoid")
    np.testing.assert_allclose(b1 + b1[::-1], 1.0, rtol=0, atol=1e-15)  # sigmoid(x) + sigmoid(-x)
    assert b1[40] == 0.5 and b2[40] == 1.0
    assert np.all((b1 > 0) & (b1 < 1)) and np.all((b2 > 0) & (b2 < 2))
    np.testing.assert_allclose(b2, 2.0 * b1, rtol=0, atol=0)
    with pytest.raises(ValueError):
        forms.prologue(np.ones((1, 4)), np.ones((1, 4)), x, "tanh")


# --- planted mistakes: each must fail one of the pins above ----------------
def _norm_then_silu(q_raw, k_raw, beta_raw, beta_map="sigmoid"):
    f = lambda x: forms.silu(x / np.linalg.norm(x, axis=-1, keepdims=True))
    return f(q_raw), f(k_raw), 1.0 / (1.0 + np.exp(-beta_raw))


def _sigmoid_for_silu(q_raw, k_raw, beta_raw, beta_map="sigmoid"):
    f = lambda x: (lambda y: y / np.linalg.norm(y, axis=-1, keepdims=True))(1 / (1 + np.exp(-x)))
    return f(q_raw), f(k_raw), 1.0 / (1.0 + np.exp(-beta_raw))


@pytest.mark.parametrize("mutant", [_norm_then_silu, _sigmoid_for_silu])
def test_pins_catch_planted_mistakes(monkeypatch, mutant):
    monkeypatch.setattr(forms, "prologue", mutant)
    caught = 0
    for pin in (test_keys_have_unit_norm_and_keep_signs,
                test_large_positive_inputs_reduce_to_plain_l2_normalisation):
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught >= 1
