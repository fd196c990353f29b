"""Pins of the CPU oracle to facts the pages and the mathematics fix.

Every ``check_*`` takes a forward function with the signature of
``oracle.fwd`` so that the same checks can also be run against deliberately
broken copies of the oracle (see ``test_oracle_mutants.py``): each plausible
mistake (a dropped term, a wrong sign or index, a transposed operand, a gate
applied at the wrong place, a readout taken before the update) must make at
least one of them fail.

Page titles used in citations:
  [DR] "08 · linear 路线（三）：delta rule 与 DPLR 统一框架"
  [DP] "DeltaProduct：通过 Householder 乘积增强线性 RNN 的状态追踪" (reading notes)
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

from oracle import forms, rel_l2

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    """Parse a ``key = values`` fixture (comment lines start with '#')."""
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            vals = [float(x) for x in val.split()]
            out[key] = vals[0] if len(vals) == 1 else np.array(vals)
    return out


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def transition(fwd, ks, betas, g=None):
    """Extract the linear map of ONE token on the state: run the oracle for a
    single token with v = 0 and h0 = I (dv = dk), so that hT = A_t * I.
    ks [n_h, dk], betas [n_h]."""
    n_h, dk = ks.shape
    q = np.zeros((1, 1, 1, dk))
    k = ks.reshape(1, 1, n_h, 1, dk)
    v = np.zeros((1, 1, n_h, 1, dk))
    beta = np.asarray(betas, float).reshape(1, 1, n_h, 1)
    gg = None if g is None else np.full((1, 1, 1), g)
    h0 = np.eye(dk).reshape(1, 1, dk, dk)
    _, hT = fwd(q, k, v, beta, gg, h0, n_h=n_h)
    return hT[0, 0]


def f32(x):
    """Round to float32: the oracle reads float32 inputs."""
    return np.asarray(x, dtype=np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
def check_single_step_forms(fwd, rng):
    """[DR] §1.1-§1.3: erase-write, Householder and gradient-step forms are the
    same update; the oracle's single step equals them."""
    dk, dv = 6, 5
    S = f32(rng.standard_normal((dk, dv)))
    k = f32(unit(rng.standard_normal(dk)))
    v = f32(rng.standard_normal(dv))
    q = f32(rng.standard_normal(dk))
    for beta in (0.0, 0.37, 1.0, 1.6, 2.0):
        b = float(np.float32(beta))
        a1 = forms.step_erase_write(S, k, v, b)
        a2 = forms.step_householder(S, k, v, b)
        a3 = forms.step_gradient(S, k, v, b)
        assert np.allclose(a1, a2, atol=1e-14, rtol=0)
        assert np.allclose(a2, a3, atol=1e-14, rtol=0)
        o, hT = fwd(q.reshape(1, 1, 1, dk), k.reshape(1, 1, 1, dk),
                    v.reshape(1, 1, 1, dv), np.full((1, 1, 1), b), None,
                    S.reshape(1, 1, dk, dv))
        assert np.allclose(hT[0, 0], a2, atol=1e-13, rtol=0)
        assert np.allclose(o[0, 0, 0], a2.T @ q, atol=1e-13, rtol=0)


def check_householder_eigenvalues(fwd, rng):
    """[DR] §1.2 / [DP] §2.4: I - beta k k^T with unit k has eigenvalue 1-beta
    along k and 1 with multiplicity dk-1."""
    dk = 7
    for beta in (0.0, 0.25, 1.0, 1.5, 2.0):
        k = unit(f32(rng.standard_normal(dk)))
        k = f32(k)
        F = transition(fwd, k.reshape(1, dk), [beta])
        ev = np.sort(np.linalg.eigvals(F).real)
        kn = k / np.linalg.norm(k)
        expect = np.sort(np.r_[1.0 - beta * (k @ k), np.ones(dk - 1)])
        assert np.allclose(ev, expect, atol=1e-6), (beta, ev, expect)
        # and the eigenvector along k
        assert np.allclose(F @ kn, (1.0 - beta * (k @ k)) * kn, atol=1e-12)


def check_exact_recall(fwd, rng):
    """[DR] §1.3 / [DP] §2.1: with beta = 1 and a unit key, the updated memory
    returns exactly v_t for k_t -- reading out with q_t = k_t gives o_t = v_t,
    whatever the previous state and gate."""
    # a rectangular and a square state (the square one would hide o = S q
    # instead of S^T q only if the state were symmetric, which it is not)
    for B, T, H, dk, dv in ((1, 9, 2, 8, 5), (2, 7, 1, 6, 6)):
        k = f32(unit(rng.standard_normal((B, T, H, dk))))
        v = f32(rng.standard_normal((B, T, H, dv)))
        beta = np.ones((B, T, H))
        g = f32(rng.uniform(0.2, 1.0, (B, T, H)))
        h0 = f32(rng.standard_normal((B, H, dk, dv)))
        o, _ = fwd(k, k, v, beta, g, h0)
        assert np.allclose(o, v, atol=5e-6), np.abs(o - v).max()


def check_nh2_closed_form(fwd, rng):
    """[DP] §2.3: for n_h = 2 the token transition is
    A = I - b1 k1 k1^T - b2 k2 k2^T + b1 b2 (k2^T k1) k2 k1^T and, with the gate
    of §2.6 applied once before the sub-steps,
    H_i = g F2 F1 H_{i-1} + F2 C1 + C2, C_j = b_j k_j v_j^T."""
    dk, dv = 5, 4
    for _ in range(3):
        k1, k2 = f32(unit(rng.standard_normal((2, dk))))
        b1, b2 = f32(rng.uniform(0, 2, 2))
        A = transition(fwd, np.stack([k1, k2]), [b1, b2])
        closed = (np.eye(dk) - b1 * np.outer(k1, k1) - b2 * np.outer(k2, k2)
                  + b1 * b2 * (k2 @ k1) * np.outer(k2, k1))
        assert np.allclose(A, closed, atol=1e-12), np.abs(A - closed).max()
        # full token with gate and writes
        v1, v2 = f32(rng.standard_normal((2, dv)))
        g = float(np.float32(rng.uniform(0.1, 1.0)))
        H0 = f32(rng.standard_normal((dk, dv)))
        F1 = np.eye(dk) - b1 * np.outer(k1, k1)
        F2 = np.eye(dk) - b2 * np.outer(k2, k2)
        expect = g * F2 @ F1 @ H0 + F2 @ (b1 * np.outer(k1, v1)) + b2 * np.outer(k2, v2)
        q = f32(rng.standard_normal(dk))
        o, hT = fwd(q.reshape(1, 1, 1, dk),
                    np.stack([k1, k2]).reshape(1, 1, 2, 1, dk),
                    np.stack([v1, v2]).reshape(1, 1, 2, 1, dv),
                    np.array([b1, b2]).reshape(1, 1, 2, 1),
                    np.full((1, 1, 1), g), H0.reshape(1, 1, dk, dv), n_h=2)
        assert np.allclose(hT[0, 0], expect, atol=1e-12)
        assert np.allclose(o[0, 0, 0], expect.T @ q, atol=1e-12)


def check_identical_keys(fwd, rng):
    """[DP] §2.4: identical keys collapse to one factor with
    beta_eff = 1 - prod_j (1 - beta_j)."""
    dk = 6
    k = f32(unit(rng.standard_normal(dk)))
    kn2 = k @ k
    for betas in ([0.3, 0.9, 1.4], [2.0, 0.5], [1.0, 1.0, 1.0, 1.0]):
        A = transition(fwd, np.tile(k, (len(betas), 1)), betas)
        # with ||k||^2 = kn2 (1 up to float32 rounding) each factor scales the
        # k direction by (1 - b kn2)
        beff = (1.0 - np.prod([1.0 - b * kn2 for b in betas])) / kn2
        assert np.allclose(A, np.eye(dk) - beff * np.outer(k, k), atol=1e-12)
        # the unit-key statement of the page
        beff_page = 1.0 - np.prod([1.0 - b for b in betas])
        assert abs(beff - beff_page) < 1e-5


def check_product_vs_sum(fwd, rng):
    """[DP] §2.5 worked example (golden fixture): two identical keys with
    beta = 2 give the identity as a product; the sum of the two rank-1 updates
    would have eigenvalue -3 along k."""
    gold = read_golden("dp_product_vs_sum.txt")
    dk = 4
    k = np.zeros(dk)
    k[1] = 1.0  # exact unit key
    b1, b2 = gold["beta"]
    A = transition(fwd, np.stack([k, k]), [b1, b2])
    assert gold["product_is_identity"] == 1.0
    assert np.allclose(A, np.eye(dk), atol=1e-15)
    summed = np.eye(dk) - b1 * np.outer(k, k) - b2 * np.outer(k, k)
    assert np.isclose(k @ summed @ k, gold["sum_eigenvalue_along_k"])


def check_orthogonal_keys(fwd, rng):
    """[DP] §2.4: mutually orthogonal keys commute; A = I - sum_j b_j k_j k_j^T,
    which is symmetric."""
    dk = 6
    ks = np.eye(dk)[[0, 3, 5]]
    betas = [0.4, 1.7, 2.0]
    A = transition(fwd, ks, betas)
    expect = np.eye(dk) - sum(b * np.outer(kk, kk) for b, kk in zip(betas, ks))
    assert np.allclose(A, expect, atol=1e-15)
    assert np.allclose(A, A.T, atol=1e-15)
    A_rev = transition(fwd, ks[::-1].copy(), betas[::-1])
    assert np.allclose(A, A_rev, atol=1e-15)


def check_rotation_120(fwd, rng):
    """[DP] §2.4 worked example (golden fixture): two beta = 2 reflections give
    the printed 120-degree rotation; three tokens return the state to start."""
    gold = read_golden("dp_rotation_120.txt")
    k1, k2 = gold["k1"], gold["k2"]
    b1, b2 = gold["beta"]
    A = transition(fwd, np.stack([k1, k2]), [b1, b2])
    expect = np.stack([gold["F2F1_row0"], gold["F2F1_row1"]])
    # k2 is read as float32, so allow its rounding (~3e-8)
    assert np.allclose(A, expect, atol=1e-7), A
    period = int(gold["period"])
    T = period
    q = np.zeros((1, T, 1, 2))
    k = np.tile(np.stack([k1, k2]), (T, 1)).reshape(1, T, 2, 1, 2)
    v = np.zeros((1, T, 2, 1, 1))
    beta = np.full((1, T, 2, 1), 2.0)
    h0 = np.array([1.0, 0.0]).reshape(1, 1, 2, 1)
    _, hT = fwd(q, k, v, beta, None, h0, n_h=2)
    assert np.allclose(hT[0, 0, :, 0], [1.0, 0.0], atol=1e-6)
    # and after one and two tokens it is NOT back (genuine period 3)
    for t in (1, 2):
        _, h = fwd(q[:, :t], k[:, :t], v[:, :t], beta[:, :t], None, h0, n_h=2)
        assert np.linalg.norm(h[0, 0, :, 0] - [1.0, 0.0]) > 1.0


def check_swap_reflection(fwd, rng):
    """[DP] §3.1 (golden fixture): k = (e_a - e_b)/sqrt(2), beta = 2, B = 0
    swaps coordinates a and b of H0 = (1..n)^T."""
    gold = read_golden("dp_swap_reflection.txt")
    n, a, b = int(gold["n"]), int(gold["a"]) - 1, int(gold["b"]) - 1
    k = np.zeros(n)
    k[a], k[b] = 1.0, -1.0
    k = k / np.sqrt(2.0)
    q = np.zeros((1, 1, 1, n))
    _, hT = fwd(q, k.reshape(1, 1, 1, n), np.zeros((1, 1, 1, 1)),
                np.full((1, 1, 1), 2.0), None,
                gold["H0"].reshape(1, 1, n, 1))
    assert np.allclose(hT[0, 0, :, 0], gold["H1"], atol=1e-6)


def check_complex_eigen_condition(fwd, rng):
    """[DP] §2.4 (Appendix A): in the plane of two unit keys with c = k1^T k2,
    tau = 2 - b1 - b2 + b1 b2 c^2, delta = (1-b1)(1-b2); F2 F1 has complex
    eigenvalues exactly when tau^2 - 4 delta < 0 (trace and determinant of the
    2x2 product)."""
    hits = [0, 0]
    for _ in range(200):
        ang = rng.uniform(0, np.pi)
        k1 = np.array([1.0, 0.0])
        k2 = f32(np.array([np.cos(ang), np.sin(ang)]))
        b1, b2 = f32(rng.uniform(0, 2, 2))
        c = k1 @ k2
        n2 = k2 @ k2
        A = transition(fwd, np.stack([k1, k2]), [b1, b2])
        # exact trace/determinant for the float32-rounded key (||k2||^2 = n2)
        tau = 2 - b1 - b2 * n2 + b1 * b2 * c * c
        delta = (1 - b1) * (1 - b2 * n2)
        assert np.isclose(np.trace(A), tau, atol=1e-12)
        assert np.isclose(np.linalg.det(A), delta, atol=1e-12)
        disc = tau * tau - 4 * delta
        if abs(disc) < 1e-9:
            continue
        ev = np.linalg.eigvals(A)
        is_complex = np.abs(ev.imag).max() > 1e-12
        assert is_complex == (disc < 0)
        hits[int(is_complex)] += 1
    assert hits[0] > 10 and hits[1] > 10


def check_stability(fwd, rng):
    """[DP] §2.5 and §2.6: for unit keys, beta in [0, 2] and g in [0, 1],
    ||A_t ... A_1||_2 <= 1 for any length; rank(A_i - g_i I) <= n_h."""
    dk = 6
    for n_h in (1, 2, 3):
        T = 12
        k = unit(rng.standard_normal((1, T, n_h, 1, dk)))
        beta = rng.uniform(0, 2, (1, T, n_h, 1))
        beta[0, 0, 0, 0] = 2.0
        g = rng.uniform(0, 1, (1, T, 1))
        h0 = np.eye(dk).reshape(1, 1, dk, dk)
        _, hT = fwd(np.zeros((1, T, 1, dk)), k, np.zeros((1, T, n_h, 1, dk)),
                    beta, g, h0, n_h=n_h)
        # keys are read as float32, so ||k||^2 = 1 +- 1e-7 per factor
        assert np.linalg.norm(hT[0, 0], 2) <= 1.0 + 2e-5
        # single token with float32 keys renormalised exactly is not possible,
        # so compare against the float32 norm bound: ||F|| <= max(1, |1-b|k|^2|)
        kk = f32(k[0, 0, :, 0])
        bb = f32(beta[0, 0, :, 0])
        A = transition(fwd, kk, bb, g=float(np.float32(g[0, 0, 0])))
        gg = float(np.float32(g[0, 0, 0]))
        assert np.linalg.matrix_rank(A - gg * np.eye(dk), tol=1e-9) <= n_h
        assert np.linalg.norm(A, 2) <= 1.0 + 1e-6


def check_reset_gate(fwd, rng):
    """[DP] §3.3: g_i = 0 resets the memory -- nothing before token i can
    influence the state or the outputs from token i on."""
    B, T, H, dk, dv, n_h = 1, 10, 1, 5, 3, 2
    t0 = 6
    k = f32(unit(rng.standard_normal((B, T, n_h, H, dk))))
    v = f32(rng.standard_normal((B, T, n_h, H, dv)))
    q = f32(rng.standard_normal((B, T, H, dk)))
    beta = f32(rng.uniform(0, 1, (B, T, n_h, H)))
    g = f32(rng.uniform(0.5, 1, (B, T, H)))
    g[:, t0] = 0.0
    h0 = f32(rng.standard_normal((B, H, dk, dv)))
    o1, s1 = fwd(q, k, v, beta, g, h0, n_h=n_h)
    k2, v2 = k.copy(), v.copy()
    k2[:, :t0] = f32(unit(rng.standard_normal(k2[:, :t0].shape)))
    v2[:, :t0] += 3.0
    o2, s2 = fwd(q, k2, v2, beta, g, None, n_h=n_h)
    assert np.array_equal(o1[:, t0:], o2[:, t0:])
    assert np.array_equal(s1, s2)
    assert not np.allclose(o1[:, :t0], o2[:, :t0])


def check_exact_rational(fwd, rng):
    """Brute force on a tiny input in exact rational arithmetic (dyadic inputs
    are exact in float32): the update of [DR] §1.2 applied token by token with
    the gate of [DP] §2.6; the oracle must agree to float64 rounding."""
    B, T, H, dk, dv, n_h = 1, 4, 1, 3, 2, 2
    den = 8

    def dy(shape):
        return rng.integers(-den, den + 1, shape) / den

    q, k, v = dy((B, T, H, dk)), dy((B, T, n_h, H, dk)), dy((B, T, n_h, H, dv))
    beta = rng.integers(0, 2 * den + 1, (B, T, n_h, H)) / den
    g = rng.integers(0, den + 1, (B, T, H)) / den
    h0 = dy((B, H, dk, dv))
    F = Fraction
    S = [[F(h0[0, 0, d, c]) for c in range(dv)] for d in range(dk)]
    outs = []
    for t in range(T):
        gt = F(g[0, t, 0])
        S = [[gt * S[d][c] for c in range(dv)] for d in range(dk)]
        for j in range(n_h):
            kk = [F(x) for x in k[0, t, j, 0]]
            vv = [F(x) for x in v[0, t, j, 0]]
            bb = F(beta[0, t, j, 0])
            # transition applied as a matrix: (I - b k k^T) S + b k v^T
            Fm = [[(F(1) if a == c else F(0)) - bb * kk[a] * kk[c]
                   for c in range(dk)] for a in range(dk)]
            S = [[sum(Fm[a][d] * S[d][c] for d in range(dk)) + bb * kk[a] * vv[c]
                  for c in range(dv)] for a in range(dk)]
        qq = [F(x) for x in q[0, t, 0]]
        outs.append([sum(S[d][c] * qq[d] for d in range(dk)) for c in range(dv)])
    o, hT = fwd(q, k, v, beta, g, h0, n_h=n_h)
    exact_o = np.array([[float(x) for x in row] for row in outs])
    exact_s = np.array([[float(x) for x in row] for row in S])
    assert np.allclose(o[0, :, 0], exact_o, rtol=0, atol=1e-13)
    assert np.allclose(hT[0, 0], exact_s, rtol=0, atol=1e-13)


def check_continuation(fwd, rng):
    """The state is the whole carried context ([DP] §2.6, [DR] §2.3): running
    T1 tokens, then T2 more from the returned state, equals running T1+T2."""
    B, T, H, dk, dv, n_h = 2, 11, 2, 4, 3, 2
    T1 = 5
    q = f32(rng.standard_normal((B, T, H, dk)))
    k = f32(unit(rng.standard_normal((B, T, n_h, H, dk))))
    v = f32(rng.standard_normal((B, T, n_h, H, dv)))
    beta = f32(rng.uniform(0, 2, (B, T, n_h, H)))
    g = f32(rng.uniform(0, 1, (B, T, H)))
    o, s = fwd(q, k, v, beta, g, None, n_h=n_h)
    oa, sa = fwd(q[:, :T1], k[:, :T1], v[:, :T1], beta[:, :T1], g[:, :T1],
                 None, n_h=n_h)
    ob, sb = fwd(q[:, T1:], k[:, T1:], v[:, T1:], beta[:, T1:], g[:, T1:],
                 sa.astype(np.float32), n_h=n_h)
    # the carried state is rounded to float32 in between: compare loosely
    assert rel_l2(np.concatenate([oa, ob], 1), o) < 1e-6
    assert rel_l2(sb, s) < 1e-6
    assert np.array_equal(oa, o[:, :T1])


def check_extended_sequence(fwd, rng):
    """[DP] §4.1: DeltaProduct equals DeltaNet run on the interleaved sequence
    of length n_h*T with the gate expanded to (g_1, 1, .., 1, g_2, ...),
    keeping each token's last sub-step output."""
    B, T, H, dk, dv, n_h = 1, 7, 1, 5, 4, 3
    q = f32(rng.standard_normal((B, T, H, dk)))
    k = f32(unit(rng.standard_normal((B, T, n_h, H, dk))))
    v = f32(rng.standard_normal((B, T, n_h, H, dv)))
    beta = f32(rng.uniform(0, 2, (B, T, n_h, H)))
    g = f32(rng.uniform(0, 1, (B, T, H)))
    o, s = fwd(q, k, v, beta, g, None, n_h=n_h)
    qx, kx, vx, bx, gx, idx = forms.extend_sequence(
        q[0, :, 0], k[0, :, :, 0], v[0, :, :, 0], beta[0, :, :, 0], g[0, :, 0], n_h)
    L = T * n_h
    ox, sx = fwd(qx.reshape(1, L, 1, dk), kx.reshape(1, L, 1, dk),
                 vx.reshape(1, L, 1, dv), bx.reshape(1, L, 1),
                 gx.reshape(1, L, 1), None, n_h=1)
    assert np.allclose(ox[0, idx, 0], o[0, :, 0], atol=1e-12)
    assert np.allclose(sx, s, atol=1e-12)
    # and the explicit-matrix token loop on the extended sequence
    orf, srf = forms.recurrent_householder(qx, kx, vx, bx, gx)
    assert np.allclose(orf[idx], o[0, :, 0], atol=1e-12)
    assert np.allclose(srf, s[0, 0], atol=1e-12)


ALL_CHECKS = [
    check_single_step_forms,
    check_householder_eigenvalues,
    check_exact_recall,
    check_nh2_closed_form,
    check_identical_keys,
    check_product_vs_sum,
    check_orthogonal_keys,
    check_rotation_120,
    check_swap_reflection,
    check_complex_eigen_condition,
    check_stability,
    check_reset_gate,
    check_exact_rational,
    check_continuation,
    check_extended_sequence,
]


# ---------------------------------------------------------------------------
# The comparison metric and the decode entry point.  These take the function
# under test (``oracle.rel_l2`` / ``oracle.step``) so that planted mistakes in
# copies of them can be run through the same checks.

def check_rel_l2(rel):
    """The metric every parity tolerance rests on (global relative L2, the
    reading of the pages' "rel err"), against values computed by hand:
    ||(3, 4.5) - (3, 4)|| / ||(3, 4)|| = 0.5 / 5; the reference is the second
    argument (||(6, 8) - (3, 4)|| / 5 = 1, the other way round 5 / 10); an
    all-zero reference gives the plain norm ||(3, 4)|| = 5; a 2x2 and a
    2x2x2 array are measured over every element, not per row."""
    assert abs(rel([3.0, 4.5], [3.0, 4.0]) - 0.1) <= 1e-15
    assert abs(rel([6.0, 8.0], [3.0, 4.0]) - 1.0) <= 1e-15
    assert abs(rel([3.0, 4.0], [6.0, 8.0]) - 0.5) <= 1e-15
    assert abs(rel([3.0, 4.0], [0.0, 0.0]) - 5.0) <= 1e-15
    assert rel([1.0, -2.0], [1.0, -2.0]) == 0.0
    ref = np.array([[1.0, 2.0], [2.0, 4.0]])                  # norm 5
    x = ref + np.array([[0.3, 0.0], [0.0, 0.4]])              # error norm 0.5
    assert abs(rel(x, ref) - 0.1) <= 1e-15
    ref3 = np.ones((2, 2, 2))                                 # norm sqrt(8)
    x3 = ref3.copy()
    x3[1, 1, 1] = 1.0 + np.sqrt(8.0) * 0.25                   # error sqrt(8) / 4
    assert abs(rel(x3, ref3) - 0.25) <= 1e-15


# exactly representable, unit norm and mutually orthogonal in float32
_K1 = np.array([0.5, 0.5, 0.5, 0.5])
_K2 = np.array([0.5, -0.5, 0.5, -0.5])


def check_step_recall(step, rng):
    """One decode step ([DR] §2.3, the recurrent form; [DP] §2.6, gate then
    n_h sub-steps).  With beta = 1 and orthogonal unit keys k1, k2 the step
    writes both values so that S^T k1 = v1 and S^T k2 = v2 exactly, whatever
    the gate and the previous state ([DR] §1.2, exact recall); the readout
    with q = k1 returns v1.  The part of the state orthogonal to both keys is
    only scaled by g, and g = 0 erases it ([DP] §3.3, the reset)."""
    dk, dv, B, H = 4, 3, 1, 2
    S0 = rng.standard_normal((B, H, dk, dv))
    v = f32(rng.standard_normal((B, 2, H, dv)))
    k = np.broadcast_to(np.stack([_K1, _K2])[None, :, None, :], (B, 2, H, dk)).copy()
    q = np.broadcast_to(_K1, (B, H, dk)).copy()
    beta = np.ones((B, 2, H))
    proj = np.eye(dk) - np.outer(_K1, _K1) - np.outer(_K2, _K2)
    for gval in (0.0, 0.5, 1.0):
        g = np.full((B, H), gval)
        out, S = step(q, k, v, beta, g, S0, n_h=2)
        for h in range(H):
            assert np.allclose(S[0, h].T @ _K1, v[0, 0, h], atol=1e-12, rtol=0)
            assert np.allclose(S[0, h].T @ _K2, v[0, 1, h], atol=1e-12, rtol=0)
            assert np.allclose(out[0, h], v[0, 0, h], atol=1e-12, rtol=0)
            assert np.allclose(proj @ S[0, h], gval * (proj @ S0[0, h]), atol=1e-12, rtol=0)


def check_step_chain(step, fwd, rng):
    """Decode calls chained through the carried state equal one forward over
    the same tokens: the state is carried in float64, never rounded, so the
    two agree to the last bit (allowed: 1e-15 relative).  Starts from a
    float64 state that float32 cannot represent."""
    B, H, dk, dv, n_h, calls = 2, 2, 5, 4, 2, 3
    S = rng.standard_normal((B, H, dk, dv)) * (1.0 + 2.0 ** -40)
    toks = []
    for _ in range(calls):
        q = f32(rng.standard_normal((B, H, dk)))
        k = f32(unit(rng.standard_normal((B, n_h, H, dk))))
        v = f32(rng.standard_normal((B, n_h, H, dv)))
        beta = f32(rng.uniform(0.0, 2.0, (B, n_h, H)))
        g = f32(rng.uniform(0.5, 1.0, (B, H)))
        toks.append((q, k, v, beta, g))
    S0 = S.copy()
    outs = []
    for (q, k, v, beta, g) in toks:
        o, S = step(q, k, v, beta, g, S, n_h=n_h)
        outs.append(o)
    Q, K, V, Bt, G = (np.stack([t[i] for t in toks], 1) for i in range(5))
    # the forward is given the carried-in state by one step with a zero
    # write (beta = 0, g = 1), which leaves it exactly unchanged
    z = np.zeros
    _, S0c = step(z((B, H, dk)), z((B, 1, H, dk)), z((B, 1, H, dv)), z((B, 1, H)),
                  None, S0, n_h=1)
    assert np.array_equal(S0c, S0)
    O, ST = fwd(Q, K, V, Bt, G, S0, n_h=n_h, state64=True)
    assert rel_l2(np.stack(outs, 1), O) <= 1e-15
    assert rel_l2(S, ST) <= 1e-15
