"""Pins of the oracle's gradients of the recurrence (``oracle.forms.
recurrent_grad``; no page states backward formulas), CPU only: central finite
differences of the forward loss through the independent float64 forms, on
tiny inputs, for every argument, and planted mistakes these pins catch."""
import numpy as np
import pytest

from oracle import forms
from pins import unit


def loss(q, k, v, beta, g, S0, dout, dST, n_h):
    # <dout, o> + <dST, S_T>, the forward written once more as a plain loop
    T = q.shape[0]
    S = np.array(S0, float)
    L = 0.0
    for t in range(T):
        if g is not None:
            S = g[t] * S
        for j in range(n_h):
            kk = k[t, j]
            S = S + beta[t, j] * np.outer(kk, v[t, j] - S.T @ kk)
        L += dout[t] @ (S.T @ q[t])
    return L + np.sum(dST * S)


def fd(f, x, eps=1e-6):
    gr = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        x0 = x[i]
        x[i] = x0 + eps
        lp = f()
        x[i] = x0 - eps
        lm = f()
        x[i] = x0
        gr[i] = (lp - lm) / (2 * eps)
    return gr


@pytest.mark.parametrize("n_h,gated", [(1, False), (1, True), (2, True), (3, False)])
def test_gradients_match_finite_differences(n_h, gated):
    rng = np.random.default_rng(40 + n_h + 3 * gated)
    T, dk, dv = 4, 3, 2
    q = rng.standard_normal((T, dk))
    k = unit(rng.standard_normal((T, n_h, dk)))
    v = rng.standard_normal((T, n_h, dv))
    beta = rng.uniform(0.1, 1.8, (T, n_h))
    g = rng.uniform(0.4, 1.0, T) if gated else None
    S0 = rng.standard_normal((dk, dv)) * 0.5
    dout = rng.standard_normal((T, dv))
    dST = rng.standard_normal((dk, dv))
    got = forms.recurrent_grad(q, k, v, beta, g, S0, dout, dST, n_h=n_h)
    f = lambda: loss(q, k, v, beta, g, S0, dout, dST, n_h)
    for name, x, gx in (("q", q, got[0]), ("k", k, got[1]), ("v", v, got[2]),
                        ("beta", beta, got[3]), ("S0", S0, got[5])):
        np.testing.assert_allclose(gx, fd(f, x), rtol=1e-6, atol=1e-7, err_msg=name)
    if gated:
        np.testing.assert_allclose(got[4], fd(f, g), rtol=1e-6, atol=1e-7, err_msg="g")
    else:
        assert got[4] is None


def test_no_state_gradient_without_a_state_loss_term_keeps_the_output_path():
    # dST = None: only the outputs carry loss; dS0 still flows through them
    rng = np.random.default_rng(47)
    T, dk, dv = 3, 2, 2
    q, k, v = rng.standard_normal((T, dk)), unit(rng.standard_normal((T, 1, dk))), rng.standard_normal((T, 1, dv))
    beta, S0, dout = rng.uniform(0, 1, (T, 1)), rng.standard_normal((dk, dv)), rng.standard_normal((T, dv))
    got = forms.recurrent_grad(q, k, v, beta, None, S0, dout, None)
    f = lambda: loss(q, k, v, beta, None, S0, dout, np.zeros((dk, dv)), 1)
    np.testing.assert_allclose(got[5], fd(f, S0), rtol=1e-6, atol=1e-7)


def _wrong_sign(*a, **kw):
    out = list(forms._recurrent_grad_ok(*a, **kw))
    out[1] = -out[1]  # dk with the wrong sign
    return tuple(out)


def _dropped_beta(*a, **kw):
    out = list(forms._recurrent_grad_ok(*a, **kw))
    out[3] = np.zeros_like(out[3])
    return tuple(out)


@pytest.mark.parametrize("mutant", [_wrong_sign, _dropped_beta])
def test_pins_catch_planted_mistakes(monkeypatch, mutant):
    monkeypatch.setattr(forms, "_recurrent_grad_ok", forms.recurrent_grad, raising=False)
    monkeypatch.setattr(forms, "recurrent_grad", mutant)
    with pytest.raises(AssertionError):
        test_gradients_match_finite_differences(2, True)


# ---- the chunked backward (forms.ut_chunk_grad) ----

def _chunk_case(seed, L, dk, dv, gated):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((L, dk))
    k = unit(rng.standard_normal((L, dk)))
    v = rng.standard_normal((L, dv))
    beta = rng.uniform(0.1, 1.8, L)
    lg = np.log(rng.uniform(0.4, 1.0, L)) if gated else None
    S0 = rng.standard_normal((dk, dv)) * 0.5
    dout = rng.standard_normal((L, dv))
    dST = rng.standard_normal((dk, dv))
    return q, k, v, beta, lg, S0, dout, dST


@pytest.mark.parametrize("L,C,gated", [(7, 4, True), (8, 4, False), (5, 8, True)])
def test_chunked_backward_matches_finite_differences(L, C, gated):
    # several chunks and a ragged tail (L = 7, C = 4), one chunk, a part chunk
    dk, dv = 3, 2
    q, k, v, beta, lg, S0, dout, dST = _chunk_case(60 + L + C, L, dk, dv, gated)
    got = forms.ut_chunk_grad(q, k, v, beta, lg, S0, dout, dST, C=C)
    f = lambda: loss(q, k[:, None], v[:, None], beta[:, None],
                     None if lg is None else np.exp(lg), S0, dout, dST, 1)
    for name, x, gx in (("q", q, got[0]), ("k", k, got[1]), ("v", v, got[2]),
                        ("beta", beta, got[3]), ("S0", S0, got[5])):
        np.testing.assert_allclose(gx, fd(f, x), rtol=1e-6, atol=1e-7, err_msg=name)
    if gated:
        # the gradient with respect to log g
        np.testing.assert_allclose(got[4], fd(f, lg), rtol=1e-6, atol=1e-7, err_msg="log g")


@pytest.mark.parametrize("L,C", [(37, 8), (33, 16), (16, 16)])
def test_chunked_backward_agrees_with_the_recurrent_gradients(L, C):
    dk, dv = 8, 6
    q, k, v, beta, lg, S0, dout, dST = _chunk_case(70 + L, L, dk, dv, True)
    g = np.exp(lg)
    ref = forms.recurrent_grad(q, k[:, None], v[:, None], beta[:, None], g, S0, dout, dST)
    got = forms.ut_chunk_grad(q, k, v, beta, lg, S0, dout, dST, C=C)
    pairs = ((got[0], ref[0]), (got[1], ref[1][:, 0]), (got[2], ref[2][:, 0]),
             (got[3], ref[3][:, 0]), (got[4], ref[4] * g), (got[5], ref[5]))
    for x, r in pairs:
        np.testing.assert_allclose(x, r, rtol=1e-10, atol=1e-12)


def _index_slip(*a, **kw):
    out = list(forms._ut_chunk_grad_ok(*a, **kw))
    out[4] = np.roll(out[4], 1)  # d log g one row off
    return tuple(out)


def _swapped_operands(*a, **kw):
    out = list(forms._ut_chunk_grad_ok(*a, **kw))
    out[0], out[1] = out[1], out[0]  # dq and dk exchanged
    return tuple(out)


@pytest.mark.parametrize("mutant", [_index_slip, _swapped_operands])
def test_chunked_pins_catch_planted_mistakes(monkeypatch, mutant):
    monkeypatch.setattr(forms, "_ut_chunk_grad_ok", forms.ut_chunk_grad, raising=False)
    monkeypatch.setattr(forms, "ut_chunk_grad", mutant)
    with pytest.raises(AssertionError):
        test_chunked_backward_matches_finite_differences(7, 4, True)


@pytest.mark.parametrize("n_h,C", [(2, 4), (3, 8)])
def test_chunked_backward_on_the_extended_sequence(n_h, C):
    # DeltaProduct ([DP] §4.1): the chunked backward on the extended sequence
    # (gate on each token's first sub-step, readout on its last) gives the
    # gradients of the token recurrence: dq from the readout rows, d log g
    # from the first sub-steps, k, v and beta per sub-step
    rng = np.random.default_rng(90 + n_h)
    T, dk, dv = 7, 4, 3
    q = rng.standard_normal((T, dk))
    k = unit(rng.standard_normal((T, n_h, dk)))
    v = rng.standard_normal((T, n_h, dv))
    beta = rng.uniform(0.1, 1.8, (T, n_h))
    g = rng.uniform(0.4, 1.0, T)
    S0 = rng.standard_normal((dk, dv)) * 0.5
    dout = rng.standard_normal((T, dv))
    dST = rng.standard_normal((dk, dv))
    ref = forms.recurrent_grad(q, k, v, beta, g, S0, dout, dST, n_h=n_h)
    qx, kx, vx, bx, gx, idx = forms.extend_sequence(q, k, v, beta, g, n_h)
    dox = np.zeros((T * n_h, dv))
    dox[idx] = dout
    got = forms.ut_chunk_grad(qx, kx, vx, bx, np.log(gx), S0, dox, dST, C=C)
    np.testing.assert_allclose(got[0][idx], ref[0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got[1].reshape(T, n_h, dk), ref[1], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got[2].reshape(T, n_h, dv), ref[2], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got[3].reshape(T, n_h), ref[3], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got[4][0::n_h], ref[4] * g, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got[5], ref[5], rtol=1e-10, atol=1e-12)
