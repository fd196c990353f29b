"""Pins of the channel-wise-gate (KDA) oracle form ``oracle.forms.
kda_recurrent`` ([DR] §1.4 family table), CPU only: the [DR] §5 DPLR
reduction of KDA (w = alpha, a = -beta k, b = alpha * k, write beta k v^T),
the reduction to Gated DeltaNet when alpha is the same on every channel (the
C oracle), the reset and the pass-through special cases, and planted
mistakes that these pins must catch."""
import numpy as np
import pytest

import oracle
from oracle import forms
from pins import f32, unit


def inputs(rng, T=12, dk=5, dv=3, n_h=1):
    q = rng.standard_normal((T, dk))
    k = unit(rng.standard_normal((T, n_h, dk)))
    v = rng.standard_normal((T, n_h, dv))
    beta = rng.uniform(0, 1.5, (T, n_h))
    alpha = rng.uniform(0.2, 1.0, (T, dk))
    S0 = rng.standard_normal((dk, dv)) * 0.5
    return q, k, v, beta, alpha, S0


def test_kda_is_the_dplr_reduction_of_the_delta_rule_page():
    # [DR] §5: KDA = DPLR with w = alpha_t, a = -beta k, b = alpha_t * k
    rng = np.random.default_rng(21)
    q, k, v, beta, alpha, S0 = inputs(rng)
    o, S = forms.kda_recurrent(q, k, v, beta, alpha, S0)
    k1, v1, b1 = k[:, 0], v[:, 0], beta[:, 0]
    o2, S2 = forms.dplr(q, alpha, -b1[:, None] * k1, alpha * k1, b1[:, None] * k1, v1, S0)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, S2, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n_h", [1, 3])
def test_channel_constant_alpha_is_gated_deltanet(n_h):
    rng = np.random.default_rng(22 + n_h)
    q, k, v, beta, alpha, S0 = inputs(rng, n_h=n_h)
    g = rng.uniform(0.3, 1.0, q.shape[0])
    alpha = np.repeat(g[:, None], q.shape[1], axis=1)
    q, k, v, beta, g, alpha, S0 = (f32(x) for x in (q, k, v, beta, g, alpha, S0))
    o, S = forms.kda_recurrent(q, k, v, beta, alpha, S0, n_h=n_h)
    T, dk = q.shape
    dv = v.shape[-1]
    o2, S2 = oracle.fwd(q.reshape(1, T, 1, dk), k.reshape(1, T, n_h, 1, dk),
                        v.reshape(1, T, n_h, 1, dv), beta.reshape(1, T, n_h, 1),
                        g.reshape(1, T, 1), S0.reshape(1, 1, dk, dv), n_h=n_h)
    np.testing.assert_allclose(o, o2[0, :, 0], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(S, S2[0, 0], rtol=1e-10, atol=1e-10)


def test_zero_gate_channel_forgets_that_row_only():
    rng = np.random.default_rng(23)
    q, k, v, beta, alpha, S0 = inputs(rng, T=1)
    alpha[0] = 1.0
    alpha[0, 2] = 0.0           # channel 2 reset, the others kept
    beta[0, 0] = 0.0            # no write: only the decay acts
    _, S = forms.kda_recurrent(q, k, v, beta, alpha, S0)
    expect = S0.copy()
    expect[2] = 0.0
    np.testing.assert_allclose(S, expect, rtol=0, atol=0)


def test_unit_gate_is_deltanet():
    rng = np.random.default_rng(24)
    q, k, v, beta, alpha, S0 = inputs(rng)
    o, S = forms.kda_recurrent(q, k, v, beta, np.ones_like(alpha), S0)
    o2, S2 = forms.recurrent_householder(q, k[:, 0], v[:, 0], beta[:, 0], None, S0)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, S2, rtol=1e-12, atol=1e-12)


# --- planted mistakes -------------------------------------------------------
def _decay_after_update(q, k, v, beta, alpha, S0=None, n_h=1):
    T, dk = q.shape
    S = np.array(S0, float)
    o = np.zeros((T, np.asarray(v).shape[-1]))
    for t in range(T):
        kk = k[t, 0]
        S = S + beta[t, 0] * np.outer(kk, v[t, 0] - S.T @ kk)
        S = alpha[t][:, None] * S
        o[t] = S.T @ q[t]
    return o, S


def _decay_on_columns(q, k, v, beta, alpha, S0=None, n_h=1):
    T, dk = q.shape
    S = np.array(S0, float)
    dv = S.shape[1]
    o = np.zeros((T, dv))
    for t in range(T):
        S = S * alpha[t][None, :dv]  # the gate on the value index
        kk = k[t, 0]
        S = S + beta[t, 0] * np.outer(kk, v[t, 0] - S.T @ kk)
        o[t] = S.T @ q[t]
    return o, S


@pytest.mark.parametrize("mutant", [_decay_after_update, _decay_on_columns])
def test_pins_catch_planted_mistakes(monkeypatch, mutant):
    monkeypatch.setattr(forms, "kda_recurrent", mutant)
    with pytest.raises(AssertionError):
        test_kda_is_the_dplr_reduction_of_the_delta_rule_page()


@pytest.mark.parametrize("n_h,C,T", [(1, 4, 12), (2, 8, 13), (3, 16, 9), (1, 64, 20)])
def test_chunked_kda_equals_the_recurrence(n_h, C, T):
    # the chunkwise form with the per-channel ratio inside the key sums (the
    # reading the CUDA-core kernel implements) is exact: several chunks, ragged
    # tails, DeltaProduct sub-steps
    rng = np.random.default_rng(30 + n_h + C)
    q, k, v, beta, alpha, S0 = inputs(rng, T=T, n_h=n_h)
    o1, S1 = forms.kda_recurrent(q, k, v, beta, alpha, S0, n_h=n_h)
    o2, S2 = forms.kda_chunk(q, k, v, beta, alpha, S0, n_h=n_h, C=C)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S2, S1, rtol=1e-12, atol=1e-12)


def test_chunked_kda_with_a_reset_inside_a_chunk():
    # alpha = 0 on some channels mid-chunk: the chunked form clamps log alpha
    # at -80 and still matches the exact recurrence
    rng = np.random.default_rng(35)
    q, k, v, beta, alpha, S0 = inputs(rng, T=10)
    alpha[3, :2] = 0.0
    alpha[6, 4] = 0.0
    o1, S1 = forms.kda_recurrent(q, k, v, beta, alpha, S0)
    o2, S2 = forms.kda_chunk(q, k, v, beta, alpha, S0, C=8)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S2, S1, rtol=1e-12, atol=1e-12)


def _channel_mean_gate(q, k, v, beta, alpha, S0=None, n_h=1, C=16):
    # a plausible slip: one gate per token (the channel mean) instead of one
    # per key channel
    a = np.repeat(np.asarray(alpha).mean(axis=1, keepdims=True), np.shape(alpha)[1], axis=1)
    return forms._kda_chunk_ok(q, k, v, beta, a, S0, n_h=n_h, C=C)


def _gate_on_last_substep(q, k, v, beta, alpha, S0=None, n_h=1, C=16):
    # another: the gate applied after a token's sub-steps (shift the tokens'
    # gates one token later, so the decay lands after the previous updates)
    a = np.concatenate([np.ones((1, np.shape(alpha)[1])), np.asarray(alpha)[:-1]])
    return forms._kda_chunk_ok(q, k, v, beta, a, S0, n_h=n_h, C=C)


@pytest.mark.parametrize("mutant", [_channel_mean_gate, _gate_on_last_substep])
def test_chunked_kda_pins_catch_planted_mistakes(monkeypatch, mutant):
    monkeypatch.setattr(forms, "_kda_chunk_ok", forms.kda_chunk, raising=False)
    monkeypatch.setattr(forms, "kda_chunk", mutant)
    with pytest.raises(AssertionError):
        test_chunked_kda_equals_the_recurrence(2, 8, 13)
