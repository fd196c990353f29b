"""The C oracle (token-by-token recurrence) against independent float64
restatements of the other forms on the pages (CPU only, tiny inputs).

Tolerances come from the agreement the pages report for these rewrites
(golden fixture ``dr_reported_agreement.txt``) with a margin of x100.
"""
import numpy as np
import pytest

import oracle
from oracle import forms, rel_l2
from pins import read_golden, unit, f32

GOLD = read_golden("dr_reported_agreement.txt")
TOL = GOLD["margin"] * max(GOLD["deltanet_chunk_vs_recurrent"],
                           GOLD["gdn_chunk_vs_recurrent"])


def head_inputs(rng, L, dk, dv, gated=True, beta_hi=1.0, g_lo=0.3):
    q = f32(rng.standard_normal((L, dk)))
    k = f32(unit(rng.standard_normal((L, dk))))
    v = f32(rng.standard_normal((L, dv)))
    beta = f32(rng.uniform(0, beta_hi, L))
    g = f32(rng.uniform(g_lo, 1.0, L)) if gated else None
    S0 = f32(rng.standard_normal((dk, dv)) * 0.5)
    return q, k, v, beta, g, S0


def run_oracle(q, k, v, beta, g, S0):
    L, dk = q.shape
    dv = v.shape[1]
    o, s = oracle.fwd(q.reshape(1, L, 1, dk), k.reshape(1, L, 1, dk),
                      v.reshape(1, L, 1, dv), beta.reshape(1, L, 1),
                      None if g is None else g.reshape(1, L, 1),
                      None if S0 is None else S0.reshape(1, 1, dk, dv))
    return o[0, :, 0], s[0, 0]


@pytest.mark.parametrize("gated", [False, True])
def test_householder_loop(gated):
    rng = np.random.default_rng(1)
    q, k, v, beta, g, S0 = head_inputs(rng, 37, 8, 6, gated, beta_hi=2.0)
    o, s = run_oracle(q, k, v, beta, g, S0)
    o2, s2 = forms.recurrent_householder(q, k, v, beta, g, S0)
    assert rel_l2(o, o2) < TOL and rel_l2(s, s2) < TOL


@pytest.mark.parametrize("C", [1, 3, 7, 16])
def test_wy_representation(C):
    rng = np.random.default_rng(2)
    q, k, v, beta, _, S0 = head_inputs(rng, 41, 8, 5, gated=False)
    o, s = run_oracle(q, k, v, beta, None, S0)
    o2, s2 = forms.wy_chunk(q, k, v, beta, S0, C)
    assert rel_l2(o, o2) < TOL and rel_l2(s, s2) < TOL


@pytest.mark.parametrize("C", [1, 7, 16, 50, 64])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("beta_hi", [1.0, 2.0])
def test_ut_chunkwise(C, gated, beta_hi):
    rng = np.random.default_rng(3 + C)
    L = 50  # ragged against 7, 16 and 64
    q, k, v, beta, g, S0 = head_inputs(rng, L, 16, 8, gated, beta_hi)
    o, s = run_oracle(q, k, v, beta, g, S0)
    lg = None if g is None else np.log(g)
    o2, s2 = forms.ut_chunk(q, k, v, beta, lg, S0, C)
    assert rel_l2(o, o2) < TOL, rel_l2(o, o2)
    assert rel_l2(s, s2) < TOL, rel_l2(s, s2)


def test_ut_chunkwise_deltaproduct_extended():
    """[DP] §4.1: the chunkwise DeltaNet form run on the extended sequence with
    the expanded gate equals the DeltaProduct oracle (readout at each token's
    last sub-step), also when token groups straddle chunk boundaries."""
    rng = np.random.default_rng(4)
    T, n_h, dk, dv = 23, 3, 8, 6
    q = f32(rng.standard_normal((1, T, 1, dk)))
    k = f32(unit(rng.standard_normal((1, T, n_h, 1, dk))))
    v = f32(rng.standard_normal((1, T, n_h, 1, dv)))
    beta = f32(2.0 * rng.uniform(0, 1, (1, T, n_h, 1)))
    g = f32(rng.uniform(0.3, 1, (1, T, 1)))
    o, s = oracle.fwd(q, k, v, beta, g, None, n_h=n_h)
    qx, kx, vx, bx, gx, idx = forms.extend_sequence(
        q[0, :, 0], k[0, :, :, 0], v[0, :, :, 0], beta[0, :, :, 0], g[0, :, 0], n_h)
    for C in (4, 16, 64):
        ox, sx = forms.ut_chunk(qx, kx, vx, bx, np.log(gx), None, C)
        assert rel_l2(ox[idx], o[0, :, 0]) < TOL
        assert rel_l2(sx, s[0, 0]) < TOL


def test_gate_zero_with_log_clamp():
    """A zero gate has log g = -inf; the chunkwise form takes log g clamped at
    -80 (e^-80 ~ 1.8e-35).  It must match the oracle's exact reset."""
    rng = np.random.default_rng(5)
    q, k, v, beta, g, S0 = head_inputs(rng, 40, 8, 8, gated=True)
    g[[3, 17, 18, 39]] = 0.0
    o, s = run_oracle(q, k, v, beta, g, S0)
    lg = np.maximum(np.log(np.maximum(g, 1e-300)), -80.0)
    o2, s2 = forms.ut_chunk(q, k, v, beta, lg, S0, 16)
    assert rel_l2(o, o2) < TOL and rel_l2(s, s2) < TOL


def test_parallel_form():
    rng = np.random.default_rng(6)
    q, k, v, beta, _, _ = head_inputs(rng, 30, 8, 5, gated=False)
    o, _ = run_oracle(q, k, v, beta, None, None)
    o2 = forms.parallel_form(q, k, v, beta)
    assert rel_l2(o, o2) < TOL


def test_dplr_reductions():
    """[DR] §5: DeltaNet is DPLR with w = 1, a = -beta k, b = k, write beta k v^T;
    Gated DeltaNet has w = alpha, a = -beta k, b = alpha k."""
    rng = np.random.default_rng(7)
    L, dk, dv = 25, 6, 4
    q, k, v, beta, g, S0 = head_inputs(rng, L, dk, dv, gated=True)
    ones = np.ones((L, dk))
    o, s = run_oracle(q, k, v, beta, None, S0)
    o2, s2 = forms.dplr(q, ones, -beta[:, None] * k, k, beta[:, None] * k, v, S0)
    assert rel_l2(o, o2) < GOLD["margin"] * GOLD["dplr_deltanet"] * 10
    assert rel_l2(s, s2) < GOLD["margin"] * GOLD["dplr_deltanet"] * 10
    o, s = run_oracle(q, k, v, beta, g, S0)
    o2, s2 = forms.dplr(q, g[:, None] * ones, -beta[:, None] * k,
                        g[:, None] * k, beta[:, None] * k, v, S0)
    assert rel_l2(o, o2) < GOLD["margin"] * GOLD["dplr_gdn"] * 10
    assert rel_l2(s, s2) < GOLD["margin"] * GOLD["dplr_gdn"] * 10


def test_product_expansion():
    rng = np.random.default_rng(8)
    q, k, v, beta, _, S0 = head_inputs(rng, 9, 5, 4, gated=False, beta_hi=2.0)
    o, s = run_oracle(q, k, v, beta, None, S0)
    o2, s2 = forms.product_expansion(q, k, v, beta, S0)
    assert rel_l2(o, o2) < TOL and rel_l2(s, s2) < TOL


def test_batched_heads_are_independent():
    """Every (b, h) head is an independent sequence: running the batch at once
    equals running each head alone (also checks the oracle's layouts)."""
    rng = np.random.default_rng(9)
    B, T, H, dk, dv, n_h = 2, 13, 3, 6, 5, 2
    q = f32(rng.standard_normal((B, T, H, dk)))
    k = f32(unit(rng.standard_normal((B, T, n_h, H, dk))))
    v = f32(rng.standard_normal((B, T, n_h, H, dv)))
    beta = f32(rng.uniform(0, 2, (B, T, n_h, H)))
    g = f32(rng.uniform(0, 1, (B, T, H)))
    h0 = f32(rng.standard_normal((B, H, dk, dv)))
    o, s = oracle.fwd(q, k, v, beta, g, h0, n_h=n_h, threads=4)
    for b in range(B):
        for h in range(H):
            o1, s1 = oracle.fwd(q[b:b+1, :, h:h+1], k[b:b+1, :, :, h:h+1],
                                v[b:b+1, :, :, h:h+1], beta[b:b+1, :, :, h:h+1],
                                g[b:b+1, :, h:h+1], h0[b:b+1, h:h+1], n_h=n_h,
                                threads=1)
            assert np.array_equal(o1[0, :, 0], o[b, :, h])
            assert np.array_equal(s1[0, 0], s[b, h])


@pytest.mark.parametrize("C", [4, 16, 64])
def test_ut_transform_gives_the_wy_vectors(C):
    """[DR] §2.1 vs §2.2: the UT transform T = (I + A)^{-1} diag(beta) of a
    chunk produces the WY vectors that the row-by-row recursion
    w_r = beta_r (k_r - sum_{i<r} w_i (k_i^T k_r)) (and the same for u with v)
    builds, W = T K and U = T V (ungated).  L is not a multiple of C: the
    padded rows of the last chunk are identity steps (T = 0 there)."""
    rng = np.random.default_rng(C)
    L, dk, dv = 2 * C + 3, 8, 5
    k = rng.standard_normal((L, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((L, dv))
    beta = rng.uniform(0.0, 2.0, L)
    Ts = forms.ut_transform(k, beta, None, C)
    assert Ts.shape == (-(-L // C), C, C)
    for n in range(Ts.shape[0]):
        s, e = n * C, min(n * C + C, L)
        w = np.zeros((e - s, dk))
        u = np.zeros((e - s, dv))
        for r in range(e - s):
            w[r] = beta[s + r] * (k[s + r] - sum(w[i] * (k[s + i] @ k[s + r]) for i in range(r)))
            u[r] = beta[s + r] * (v[s + r] - sum(u[i] * (k[s + i] @ k[s + r]) for i in range(r)))
        T = Ts[n][: e - s, : e - s]
        assert np.allclose(T @ k[s:e], w, atol=1e-12, rtol=0)
        assert np.allclose(T @ v[s:e], u, atol=1e-12, rtol=0)
        assert not Ts[n][e - s:].any() and not Ts[n][:, e - s:].any()


def test_ut_transform_special_cases():
    """Orthogonal keys give A = 0, so T = diag(beta); beta = 0 gives T = 0;
    a gate of 0 at row r ([DP] §3.3) cuts every coupling across r
    (Gam_ij = 0 for j < r <= i), so T is block diagonal there."""
    C, dk = 8, 8
    k = np.eye(dk)
    beta = np.linspace(0.1, 1.9, C)
    assert np.array_equal(forms.ut_transform(k, beta, None, C)[0], np.diag(beta))
    assert not forms.ut_transform(k, np.zeros(C), None, C).any()
    rng = np.random.default_rng(3)
    k = rng.standard_normal((C, dk))
    lg = np.zeros(C)
    lg[5] = -1e4  # log g far below where exp underflows to 0 (g = 0)
    T = forms.ut_transform(k, np.ones(C), lg, C)[0]
    assert not T[5:, :5].any()
    assert np.allclose(T[:5, :5], forms.ut_transform(k[:5], np.ones(5), None, 5)[0])


# --- diagnostics on the outputs: the attention map and the effective rank ---
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("L", [1, 9, 64])
def test_attention_map_reproduces_the_recurrence(gated, L):
    # [DR] §2.4: o_i = sum_j A_ij v_j for a zero initial state -- pinned to
    # the token-by-token C oracle
    rng = np.random.default_rng(40 + L)
    q, k, v, beta, g, _ = head_inputs(rng, L, 8, 5, gated, beta_hi=2.0)
    o, _ = run_oracle(q, k, v, beta, g, None)
    A = forms.attention_map(q, k, beta, None if g is None else np.log(g.astype(np.float64)))
    assert rel_l2(A @ v, o) < TOL


def test_attention_map_structure():
    # causal (zero above the diagonal); A_ii = beta_i (q_i . k_i) because T is
    # lower triangular with T_ii = beta_i; ungated it is the map of the
    # fully parallel form
    rng = np.random.default_rng(43)
    q, k, v, beta, g, _ = head_inputs(rng, 20, 6, 4, True)
    A = forms.attention_map(q, k, beta, np.log(g.astype(np.float64)))
    assert np.all(np.triu(A, 1) == 0.0)
    qk = np.einsum("id,id->i", q.astype(np.float64), k.astype(np.float64))
    assert np.allclose(np.diag(A), beta * qk, rtol=1e-12, atol=1e-14)
    A0 = forms.attention_map(q, k, beta)
    assert rel_l2(A0 @ v, forms.parallel_form(q, k, v, beta)) < TOL


def test_effective_rank_closed_forms():
    # [DP] §4.6: erank = exp(entropy of sigma / sum sigma)
    er = forms.effective_rank
    assert abs(er(np.eye(7)) - 7.0) < 1e-12                       # 7 equal singular values
    rng = np.random.default_rng(44)
    a, b = rng.standard_normal(6), rng.standard_normal(9)
    assert abs(er(np.outer(a, b)) - 1.0) < 1e-12                  # rank one
    sv = np.array([1.0, 1.0, 2.0])                                # p = 1/4, 1/4, 1/2
    want = np.exp(-(0.5 * np.log(0.25) + 0.5 * np.log(0.5)))      # = 2^(3/2)
    assert abs(want - 2.0 ** 1.5) < 1e-12
    assert abs(er(np.diag(sv)) - want) < 1e-12
    # invariant under orthogonal maps on either side and under scaling
    U, _ = np.linalg.qr(rng.standard_normal((3, 3)))
    V, _ = np.linalg.qr(rng.standard_normal((3, 3)))
    assert abs(er(-3.5 * U @ np.diag(sv) @ V.T) - want) < 1e-12
    assert er(np.zeros((4, 5))) == 0.0                            # the definition does not apply


def test_effective_rank_bounds():
    # 1 <= erank <= rank for nonzero matrices
    rng = np.random.default_rng(45)
    for r in (1, 2, 5, 8):
        M = rng.standard_normal((8, r)) @ rng.standard_normal((r, 10))
        e = forms.effective_rank(M)
        assert 1.0 - 1e-12 <= e <= r + 1e-9
