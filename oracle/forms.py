"""Independent float64 restatements of the forms the pages give -- TEST
INFRASTRUCTURE ONLY (see the package docstring).

Each function works on ONE head (no batch/head axes) and follows one passage.
They are written from the mathematics, not from the printed listings, and are
used on tiny inputs to pin the C oracle (``oracle.fwd``), which implements only
the token-by-token recurrence.

Page titles used in citations:
  [DR] "08 · linear 路线（三）：delta rule 与 DPLR 统一框架" (llm-infra-atlas)
  [DP] "DeltaProduct：通过 Householder 乘积增强线性 RNN 的状态追踪" (reading notes)

Conventions: the state S is [dk, dv]; the readout is o = S^T q after the
update; keys are not normalised here.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


# --------------------------------------------------------------------------
# single-step forms ([DR] section 1)
# --------------------------------------------------------------------------
def step_erase_write(S, k, v, beta):
    """[DR] §1.1 erase-write view: erase the value stored under k, then write
    the interpolation beta*v + (1-beta)*v_old."""
    v_old = S.T @ k
    v_new = beta * v + (1.0 - beta) * v_old
    return S - np.outer(k, v_old) + np.outer(k, v_new)


def step_householder(S, k, v, beta):
    """[DR] §1.2 simplified form: S' = (I - beta k k^T) S + beta k v^T."""
    F = np.eye(len(k)) - beta * np.outer(k, k)
    return F @ S + beta * np.outer(k, v)


def step_gradient(S, k, v, beta):
    """[DR] §1.3 online-GD view: one gradient step with learning rate beta on
    L(S) = 1/2 ||S^T k - v||^2, whose gradient is k (S^T k - v)^T."""
    grad = np.outer(k, S.T @ k - v)
    return S - beta * grad


# --------------------------------------------------------------------------
# DeltaProduct algebra ([DP] sections 2.2-2.6)
# --------------------------------------------------------------------------
def householder_factor(k, beta):
    """F = I - beta k k^T ([DP] §2.2)."""
    return np.eye(len(k)) - beta * np.outer(k, k)


def householder_product(ks, betas):
    """A = F_{n_h} ... F_2 F_1: earlier factors sit on the right ([DP] §2.3)."""
    A = np.eye(ks.shape[1])
    for kj, bj in zip(ks, betas):
        A = householder_factor(kj, bj) @ A
    return A


def write_term(ks, vs, betas):
    """B = sum_j F_{n_h} ... F_{j+1} C_j with C_j = beta_j k_j v_j^T ([DP] §2.3)."""
    n = len(betas)
    Bm = np.zeros((ks.shape[1], vs.shape[1]))
    for j in range(n):
        Cj = betas[j] * np.outer(ks[j], vs[j])
        for i in range(j + 1, n):
            Cj = householder_factor(ks[i], betas[i]) @ Cj
        Bm += Cj
    return Bm


def extend_sequence(q, k, v, beta, g, n_h):
    """[DP] §4.1 extended sequence: interleave the n_h keys/values of every
    token into one sequence of length n_h*T; the gate becomes
    (g_1, 1, ..., 1, g_2, 1, ...), applied once per original token; only the
    last sub-step of each token is read out.

    q [T,dk], k [T,n_h,dk], v [T,n_h,dv], beta [T,n_h], g [T] or None.
    Returns (qx [L,dk], kx [L,dk], vx [L,dv], bx [L], gx [L], readout_idx [T]).
    """
    T, dk = q.shape
    L = T * n_h
    kx = k.reshape(L, dk)
    vx = v.reshape(L, v.shape[-1])
    bx = beta.reshape(L)
    gx = np.ones(L)
    if g is not None:
        gx[0::n_h] = g
    qx = np.repeat(q, n_h, axis=0)
    idx = np.arange(T) * n_h + (n_h - 1)
    return qx, kx, vx, bx, gx, idx


# --------------------------------------------------------------------------
# sequence forms for DeltaNet / Gated DeltaNet (one step per row)
# --------------------------------------------------------------------------
def recurrent_householder(q, k, v, beta, g=None, S0=None):
    """Token loop written with explicit transition matrices:
    S_t = g_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T, o_t = S_t^T q_t
    ([DR] §1.2 and §3; the scalar gate commutes with the Householder factor)."""
    L, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((L, dv))
    for t in range(L):
        gt = 1.0 if g is None else g[t]
        S = gt * (householder_factor(k[t], beta[t]) @ S) + beta[t] * np.outer(k[t], v[t])
        o[t] = S.T @ q[t]
    return o, S


def wy_chunk(q, k, v, beta, S0=None, C=16):
    """[DR] §2.1 WY representation, ungated.  Inside a chunk starting from
    state S0, the product of Householder factors is I - sum_i k_i w_i^T and the
    accumulated writes are sum_i k_i u_i^T, with
        w_r = beta_r (k_r - sum_{i<r} w_i (k_i^T k_r)),
        u_r = beta_r (v_r - sum_{i<r} u_i (k_i^T k_r)),
    so S_r = S0 + sum_{i<=r} k_i (u_i - S0^T w_i)^T.  Recursions run row by row."""
    L, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((L, dv))
    for s in range(0, L, C):
        e = min(s + C, L)
        n = e - s
        w = np.zeros((n, dk))
        u = np.zeros((n, dv))
        for r in range(n):
            kr = k[s + r]
            w_acc = kr.copy()
            u_acc = v[s + r].copy()
            for i in range(r):
                c = k[s + i] @ kr
                w_acc -= w[i] * c
                u_acc -= u[i] * c
            w[r] = beta[s + r] * w_acc
            u[r] = beta[s + r] * u_acc
        for r in range(n):
            Sr = S.copy()
            for i in range(r + 1):
                Sr += np.outer(k[s + i], u[i] - S.T @ w[i])
            o[s + r] = Sr.T @ q[s + r]
        Snew = S.copy()
        for i in range(n):
            Snew += np.outer(k[s + i], u[i] - S.T @ w[i])
        S = Snew
    return o, S


def ut_transform(k, beta, log_g=None, C=16):
    """[DR] §2.2 (the UT transform) with the gated decay of §3, for every
    chunk of one sequence: with gc the inclusive cumulative log gate of the
    chunk and Gam_ij = exp(gc_i - gc_j) (i > j),
        A = strictLower(diag(beta) (Gam * K K^T)),  T = (I + A)^{-1} diag(beta)
    solved as a unit lower triangular system.  A ragged tail is padded with
    identity steps (k = 0, beta = 0, log g = 0).  k [L,dk], beta [L],
    log_g [L] or None.  Returns T [NT, C, C] (float64)."""
    L, dk = k.shape
    if log_g is None:
        log_g = np.zeros(L)
    NT = -(-L // C)
    pad = NT * C - L
    K = np.concatenate([k, np.zeros((pad, dk))]) if pad else np.asarray(k, float)
    bt = np.concatenate([np.asarray(beta, float), np.zeros(pad)])
    lg = np.concatenate([np.asarray(log_g, float), np.zeros(pad)])
    strict = np.tril(np.ones((C, C), dtype=bool), -1)
    out = np.zeros((NT, C, C))
    for n in range(NT):
        sl = slice(n * C, (n + 1) * C)
        Kc, bc = K[sl], bt[sl]
        gc = np.cumsum(lg[sl])
        diff = np.where(strict, gc[:, None] - gc[None, :], -np.inf)  # mask before exp
        A = np.where(strict, bc[:, None] * (Kc @ Kc.T) * np.exp(diff), 0.0)
        out[n] = solve_triangular(np.eye(C) + A, np.diag(bc), lower=True,
                                  unit_diagonal=True)
    return out


def ut_chunk(q, k, v, beta, log_g=None, S0=None, C=16):
    """[DR] §2.2-§2.3 (UT transform + chunkwise algorithm) and §3 (the gated
    chunkwise form with the within-chunk cumulative decay).  Per chunk:
        gc_r   = sum_{e<=r} log g_e          (restarts every chunk, inclusive)
        Gam_ij = exp(gc_i - gc_j) for j <= i, else 0   (masked BEFORE exp)
        A      = strictLower(diag(beta) (Gam * K K^T))
        T      = (I + A)^{-1} diag(beta)      (unit lower triangular solve)
        W      = T (K * exp(gc)),  U = T V
        Vt     = U - W S                      (pseudo-values)
        O      = (Q * exp(gc)) S + (Q K^T * Gam) Vt
        S     <- exp(gc_C) S + (K * exp(gc_C - gc))^T Vt
    A ragged tail is padded with identity steps (k = 0, v = 0, beta = 0,
    log g = 0), which leave the state unchanged."""
    L, dk = k.shape
    dv = v.shape[1]
    if log_g is None:
        log_g = np.zeros(L)
    NT = -(-L // C)
    Lp = NT * C
    pad = Lp - L

    def padrows(x):
        return np.concatenate([x, np.zeros((pad,) + x.shape[1:])]) if pad else x

    Q, K, V = padrows(q), padrows(k), padrows(v)
    bt, lg = padrows(np.asarray(beta, float)), padrows(np.asarray(log_g, float))
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((Lp, dv))
    incl = np.tril(np.ones((C, C), dtype=bool))
    Ts = ut_transform(K, bt, lg, C)
    for n in range(NT):
        sl = slice(n * C, (n + 1) * C)
        Kc, Vc, Qc = K[sl], V[sl], Q[sl]
        gc = np.cumsum(lg[sl])
        diff = np.where(incl, gc[:, None] - gc[None, :], -np.inf)
        Gam = np.exp(diff)
        Tm = Ts[n]
        W = Tm @ (Kc * np.exp(gc)[:, None])
        U = Tm @ Vc
        Vt = U - W @ S
        o[sl] = (Qc * np.exp(gc)[:, None]) @ S + ((Qc @ Kc.T) * Gam) @ Vt
        S = np.exp(gc[-1]) * S + (Kc * np.exp(gc[-1] - gc)[:, None]).T @ Vt
    return o[:L], S


def parallel_form(q, k, v, beta):
    """[DR] §2.4 fully parallel form (ungated, zero initial state): the whole
    sequence is one block, T = (I + strictLower(diag(beta) K K^T))^{-1} diag(beta),
    and the attention-like matrix is (Q K^T * M) T with M the causal mask
    including the diagonal; o = (Q K^T * M) T V."""
    L = k.shape[0]
    A = np.tril(beta[:, None] * (k @ k.T), -1)
    Tm = solve_triangular(np.eye(L) + A, np.diag(beta), lower=True,
                          unit_diagonal=True)
    Amap = np.tril(q @ k.T) @ Tm
    return Amap @ v


def attention_map(q, k, beta, log_g=None):
    """[DR] §2.4, the fully parallel form, with the gated decay of §3: for a
    sequence of L steps processed as one block (zero initial state), the
    L x L matrix A with o_i = sum_j A_ij v_j,
        A = (Q K^T * Gam * M) T,   T = (I + strictLower(diag(beta) (Gam * K K^T)))^{-1} diag(beta)
    with Gam_ij = exp(gc_i - gc_j) (gc the inclusive cumulative log gate) and
    M the causal mask including the diagonal.  q, k [L, dk]; beta [L];
    log_g [L] or None.  Returns A [L, L] (float64)."""
    L = k.shape[0]
    if log_g is None:
        log_g = np.zeros(L)
    Tm = ut_transform(np.asarray(k, float), beta, log_g, C=L)[0]
    gc = np.cumsum(np.asarray(log_g, float))
    incl = np.tril(np.ones((L, L), dtype=bool))
    Gam = np.exp(np.where(incl, gc[:, None] - gc[None, :], -np.inf))  # mask before exp
    return ((np.asarray(q, float) @ np.asarray(k, float).T) * Gam) @ Tm


def effective_rank(Hm):
    """[DP] §4.6, the effective rank of a matrix state: with sigma_k its
    singular values and p_k = sigma_k / sum_j sigma_j,
        erank(H) = exp(-sum_k p_k log p_k)     (0 log 0 = 0).
    The definition does not apply to H = 0; that case returns 0."""
    sv = np.linalg.svd(np.asarray(Hm, dtype=np.float64), compute_uv=False)
    tot = sv.sum()
    if tot == 0.0:
        return 0.0
    p = sv[sv > 0] / tot
    return float(np.exp(-np.sum(p * np.log(p))))


def dplr(q, w, a, b, kk, vv, S0=None):
    """[DR] §5 DPLR loop: S_t = (Diag(w_t) + a_t b_t^T) S_{t-1} + kk_t vv_t^T,
    o_t = S_t^T q_t.  b_t^T acts on the UNdecayed previous state."""
    L, dk = q.shape
    dv = vv.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((L, dv))
    for t in range(L):
        S = w[t][:, None] * S + np.outer(a[t], b[t] @ S) + np.outer(kk[t], vv[t])
        o[t] = S.T @ q[t]
    return o, S


def product_expansion(q, k, v, beta, S0=None):
    """[DR] §2, the intra-chunk expansion (GDN paper Eq. 3), materialising the
    dk x dk products explicitly -- the naive O(d^2) per step form:
        P^r = prod_{i=1..r} (I - beta_i k_i k_i^T)   (left to right),
        H^r = sum_i beta_i v_i k_i^T prod_{j=i+1..r} (I - beta_j k_j k_j^T),
    written for a [dv, dk] state; transposed to [dk, dv] it reads
    S^r = (P^r)^T S0 + (H^r)^T.  The whole sequence is one block."""
    L, dk = k.shape
    dv = v.shape[1]
    S0 = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((L, dv))
    I = np.eye(dk)
    S = S0
    for r in range(L):
        P = I.copy()
        for i in range(r + 1):
            P = P @ (I - beta[i] * np.outer(k[i], k[i]))
        Hm = np.zeros((dv, dk))
        for i in range(r + 1):
            term = beta[i] * np.outer(v[i], k[i])
            for j in range(i + 1, r + 1):
                term = term @ (I - beta[j] * np.outer(k[j], k[j]))
            Hm += term
        S = P.T @ S0 + Hm.T
        o[r] = S.T @ q[r]
    return o, S


# --------------------------------------------------------------------------
# input prologue ([DP] §2.2; [DR] §3 layer design)
# --------------------------------------------------------------------------
def silu(x):
    """psi of [DP] §2.2 (SiLU): x * sigmoid(x)."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def prologue(q_raw, k_raw, beta_raw, beta_map="sigmoid"):
    """The inputs of the recurrence from raw projections, [DP] §2.2: each key
    (and, per the [DR] §3 layer design, each query) is psi(.) / ||psi(.)||_2
    over the key dimension with psi = SiLU, and beta = phi(.) with phi =
    sigmoid, or 2 sigmoid (so that beta reaches (0, 2): reflections).  The
    last axis of q_raw and k_raw is the key dimension; beta_raw is
    elementwise.  Reading: a vector whose SiLU is all zero (it has no
    direction) maps to the zero vector."""
    def unit(x):
        y = silu(x)
        n = np.sqrt(np.sum(y * y, axis=-1, keepdims=True))
        return np.divide(y, n, out=np.zeros_like(y), where=n > 0)
    b = 1.0 / (1.0 + np.exp(-np.asarray(beta_raw, dtype=np.float64)))
    if beta_map == "2sigmoid":
        b = 2.0 * b
    elif beta_map != "sigmoid":
        raise ValueError(f"beta_map {beta_map!r} is not 'sigmoid' or '2sigmoid'")
    return unit(q_raw), unit(k_raw), b


# --------------------------------------------------------------------------
# channel-wise gate (KDA; [DR] §1.4 family table and §5 DPLR reductions)
# --------------------------------------------------------------------------
def kda_recurrent(q, k, v, beta, alpha, S0=None, n_h=1):
    """The KDA recurrence of [DR] §1.4 with a per-channel gate, for one head:
        S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
        o_t = S_t^T q_t,
    the decay applied first, then the delta update on the decayed state.
    alpha_t (a vector over the key dimension) decays the rows of S.  With
    n_h > 1 ([DP] §2.6) the gate acts once per token, before its n_h
    sub-steps, and the readout follows the last one.
    Shapes: q [T, dk]; k [T, n_h, dk]; v [T, n_h, dv]; beta [T, n_h];
    alpha [T, dk]; S0 [dk, dv] or None."""
    q = np.asarray(q, float)
    k = np.asarray(k, float).reshape(q.shape[0], n_h, q.shape[1])
    v = np.asarray(v, float)
    v = v.reshape(q.shape[0], n_h, v.shape[-1])
    beta = np.asarray(beta, float).reshape(q.shape[0], n_h)
    alpha = np.asarray(alpha, float)
    T, dk = q.shape
    dv = v.shape[-1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, dv))
    for t in range(T):
        S = alpha[t][:, None] * S
        for j in range(n_h):
            kk = k[t, j]
            S = S + beta[t, j] * np.outer(kk, v[t, j] - S.T @ kk)
        o[t] = S.T @ q[t]
    return o, S



def kda_chunk(q, k, v, beta, alpha, S0=None, n_h=1, C=16):
    """The chunkwise form of the channel-wise gate: the gated chunkwise
    algorithm of [DR] §2.3 and §3 (which that page states for the whole delta
    family, KDA included) with the scalar cumulative log gate replaced by one
    per key channel, gc [C, dk], so that every decay ratio moves inside the
    sum over the key dimension:
        A_rj = beta_r sum_d k_rd k_jd exp(gc_rd - gc_jd)      (r > j)
        P_rj = sum_d q_rd k_jd exp(gc_rd - gc_jd)             (j <= r)
        T    = (I + A)^{-1} diag(beta),  W = T (K * exp(gc)),  U = T V
        Vt   = U - W S,  O = (Q * exp(gc)) S + P Vt
        S   <- Diag(exp(gc_C)) S + (K * exp(gc_C - gc))^T Vt
    run on the [DP] §4.1 extended sequence (alpha on each token's first
    sub-step, readout on its last).  The ratio is formed only for j <= r (mask
    before the exponential), so no exponent is positive.  Shapes as
    kda_recurrent; returns o [T, dv] and the final state (float64)."""
    q = np.asarray(q, float)
    T, dk = q.shape
    k = np.asarray(k, float).reshape(T, n_h, dk)
    v = np.asarray(v, float)
    v = v.reshape(T, n_h, v.shape[-1])
    dv = v.shape[-1]
    L = T * n_h
    K, V = k.reshape(L, dk), v.reshape(L, dv)
    bt = np.asarray(beta, float).reshape(L)
    lg = np.zeros((L, dk))
    with np.errstate(divide="ignore"):
        # log alpha clamped at -80, so that alpha = 0 (a reset of that row)
        # stays finite: exp(-80) is below float64 resolution next to 1
        lg[0::n_h] = np.maximum(np.log(np.asarray(alpha, float)), -80.0)
    Q = np.zeros((L, dk))
    Q[n_h - 1::n_h] = q
    NT = -(-L // C)
    pad = NT * C - L
    if pad:
        K, V, Q, lg = (np.concatenate([x, np.zeros((pad,) + x.shape[1:])]) for x in (K, V, Q, lg))
        bt = np.concatenate([bt, np.zeros(pad)])
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((NT * C, dv))
    strict = np.tril(np.ones((C, C), dtype=bool), -1)
    incl = np.tril(np.ones((C, C), dtype=bool))
    for n in range(NT):
        sl = slice(n * C, (n + 1) * C)
        Kc, Vc, Qc, bc = K[sl], V[sl], Q[sl], bt[sl]
        gc = np.cumsum(lg[sl], axis=0)                       # [C, dk]
        # ratio[r, j, d] = exp(gc_rd - gc_jd), formed only where j <= r
        diff = np.where(incl[:, :, None], gc[:, None, :] - gc[None, :, :], -np.inf)
        ratio = np.exp(diff)
        A = np.where(strict, bc[:, None] * np.einsum("rd,jd,rjd->rj", Kc, Kc, ratio), 0.0)
        P = np.einsum("rd,jd,rjd->rj", Qc, Kc, ratio)
        Tm = solve_triangular(np.eye(C) + A, np.diag(bc), lower=True, unit_diagonal=True)
        W = Tm @ (Kc * np.exp(gc))
        Vt = Tm @ Vc - W @ S
        o[sl] = (Qc * np.exp(gc)) @ S + P @ Vt
        S = np.exp(gc[-1])[:, None] * S + (Kc * np.exp(gc[-1][None, :] - gc)).T @ Vt
    return o[n_h - 1:L:n_h], S


# --------------------------------------------------------------------------
# gradients of the recurrence (no page gives them: float64 autograd)
# --------------------------------------------------------------------------
def recurrent_grad(q, k, v, beta, g, S0, dout, dST=None, n_h=1):
    """Gradients of L = <dout, o> + <dST, S_T> through the recurrence of
    [DP] §2.6 (gate once per token, then n_h delta sub-steps, readout after
    the last), for one head, by float64 reverse-mode autograd of a plain
    loop (the pages state no backward formulas).
    Shapes: q [T, dk]; k [T, n_h, dk]; v [T, n_h, dv]; beta [T, n_h];
    g [T] or None; S0 [dk, dv] or None; dout [T, dv]; dST [dk, dv] or None.
    Returns dq, dk, dv, dbeta, dg (None without g), dS0 as NumPy arrays."""
    import torch
    f64 = lambda x: torch.tensor(np.asarray(x, dtype=np.float64), requires_grad=True)
    T, dk = np.asarray(q).shape
    dv = np.asarray(v).shape[-1]
    tq = f64(q)
    tk = f64(np.asarray(k, float).reshape(T, n_h, dk))
    tv = f64(np.asarray(v, float).reshape(T, n_h, dv))
    tb = f64(np.asarray(beta, float).reshape(T, n_h))
    tg = None if g is None else f64(g)
    tS0 = f64(np.zeros((dk, dv)) if S0 is None else S0)
    S = tS0
    outs = []
    for t in range(T):
        if tg is not None:
            S = tg[t] * S
        for j in range(n_h):
            kk = tk[t, j]
            S = S + tb[t, j] * torch.outer(kk, tv[t, j] - S.T @ kk)
        outs.append(S.T @ tq[t])
    o = torch.stack(outs)
    loss = (o * torch.as_tensor(np.asarray(dout, dtype=np.float64))).sum()
    if dST is not None:
        loss = loss + (S * torch.as_tensor(np.asarray(dST, dtype=np.float64))).sum()
    loss.backward()
    grad = lambda x: None if x is None else x.grad.detach().numpy().copy()
    return grad(tq), grad(tk), grad(tv), grad(tb), grad(tg), grad(tS0)


def ut_chunk_grad(q, k, v, beta, log_g=None, S0=None, dout=None, dST=None, C=16):
    """The chunked backward: gradients of L = <dout, o> + <dST, S_T> through
    ut_chunk ([DR] §2.2-§2.3 with the §3 gate), one chunk at a time in
    reverse, by differentiating each chunk's matrix products (the pages state
    no backward formulas; this is the chain rule applied to the chunkwise
    form, written out by hand).  With the forward quantities of a chunk
    (gamma = exp(gc), gamma_C its last entry, Qg = Q * gamma, Kg = K * gamma,
    Kd = K * gamma_C / gamma, P = (Q K^T) * Gam * M, X = (I + A)^{-1},
    T = X diag(beta), W = T Kg, U = T V, Vt = U - W S) and dS the gradient
    arriving at the chunk's end state:
        dVt = Kd dS + P^T dO;   dKd = Vt dS^T;   d gamma_C = <S, dS>
        dS_prev = gamma_C dS + Qg^T dO - W^T dVt
        dQg = dO S^T;  dP = (dO Vt^T) * M
        dT = dVt V^T - dVt S^T Kg^T;  dV = T^T dVt;  dKg = -T^T dVt S^T
        dX = dT diag(beta);  dbeta_j = sum_i X_ij dT_ij;  dA = -(X^T dX X^T) * M_strict
    then A, P, Qg, Kg and Kd give dK, dQ, dbeta and the gradient of every
    exponential of gc, and d log_g is the reverse cumulative sum of dgc within
    the chunk.  Shapes and padding as ut_chunk (n_h = 1: every row is read
    out).  Returns dq, dk, dv, dbeta, dlog_g, dS0 (float64)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    L, dk = k.shape
    dv = v.shape[1]
    log_g = np.zeros(L) if log_g is None else np.asarray(log_g, dtype=np.float64)
    dout = np.zeros((L, dv)) if dout is None else np.asarray(dout, dtype=np.float64)
    NT = -(-L // C)
    Lp = NT * C
    pad = Lp - L

    def padrows(x):
        return np.concatenate([x, np.zeros((pad,) + x.shape[1:])]) if pad else x

    Q, K, V, dO = padrows(q), padrows(k), padrows(v), padrows(dout)
    bt, lg = padrows(np.asarray(beta, dtype=np.float64)), padrows(log_g)
    strict = np.tril(np.ones((C, C), dtype=bool), -1)
    incl = np.tril(np.ones((C, C), dtype=bool))
    # forward: the state at the start of every chunk
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, dtype=np.float64)
    starts = []
    Ts = ut_transform(K, bt, lg, C)
    for n in range(NT):
        sl = slice(n * C, (n + 1) * C)
        starts.append(S)
        gc = np.cumsum(lg[sl])
        Kc, Vc = K[sl], V[sl]
        Vt = Ts[n] @ Vc - (Ts[n] @ (Kc * np.exp(gc)[:, None])) @ S
        S = np.exp(gc[-1]) * S + (Kc * np.exp(gc[-1] - gc)[:, None]).T @ Vt
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    dB, dLG = np.zeros(Lp), np.zeros(Lp)
    dS = np.zeros((dk, dv)) if dST is None else np.array(dST, dtype=np.float64)
    for n in reversed(range(NT)):
        sl = slice(n * C, (n + 1) * C)
        S = starts[n]
        Qc, Kc, Vc, dOc, bc = Q[sl], K[sl], V[sl], dO[sl], bt[sl]
        gc = np.cumsum(lg[sl])
        gam, gC = np.exp(gc), np.exp(gc[-1])
        dec = np.exp(gc[-1] - gc)
        Gam = np.exp(np.where(incl, gc[:, None] - gc[None, :], -np.inf))
        KK, QK = Kc @ Kc.T, Qc @ Kc.T
        A = np.where(strict, bc[:, None] * Gam * KK, 0.0)
        X = solve_triangular(np.eye(C) + A, np.eye(C), lower=True, unit_diagonal=True)
        Tm = X * bc[None, :]
        Qg, Kg, Kd = Qc * gam[:, None], Kc * gam[:, None], Kc * dec[:, None]
        W = Tm @ Kg
        Vt = Tm @ Vc - W @ S
        P = QK * Gam
        # state update S' = gamma_C S + Kd^T Vt
        dgC = np.sum(S * dS)
        dKd = Vt @ dS.T
        dVt = Kd @ dS
        dSp = gC * dS
        # readout O = Qg S + P Vt
        dQg = dOc @ S.T
        dSp += Qg.T @ dOc
        dP = np.where(incl, dOc @ Vt.T, 0.0)
        dVt += P.T @ dOc
        # Vt = U - W S, U = T V, W = T Kg
        dW = -dVt @ S.T
        dSp -= W.T @ dVt
        dT = dVt @ Vc.T + dW @ Kg.T
        dV[sl] = Tm.T @ dVt
        dKg = Tm.T @ dW
        # T = X diag(beta), X = (I + A)^{-1}
        dX = dT * bc[None, :]
        dbeta = np.sum(X * dT, axis=0)
        dA = np.where(strict, -(X.T @ dX @ X.T), 0.0)
        # A_ij = beta_i Gam_ij (k_i . k_j), i > j
        dbeta += np.sum(dA * Gam * KK, axis=1)
        E = dA * Gam * bc[:, None]
        dKc = E @ Kc + E.T @ Kc
        dGam = dA * bc[:, None] * KK
        # P_ij = (q_i . k_j) Gam_ij, j <= i
        F = dP * Gam
        dQc = F @ Kc
        dKc += F.T @ Qc
        dGam += dP * QK
        # the scaled copies of Q and K
        dQc += dQg * gam[:, None]
        dKc += dKg * gam[:, None] + dKd * dec[:, None]
        dgam = np.sum(dQg * Qc, axis=1) + np.sum(dKg * Kc, axis=1)
        ddec = np.sum(dKd * Kc, axis=1)
        # every exponential of gc
        dgc = dgam * gam - ddec * dec
        dgc[-1] += dgC * gC + np.sum(ddec * dec)
        Z = np.where(incl, dGam * Gam, 0.0)
        dgc += Z.sum(axis=1) - Z.sum(axis=0)
        dLG[sl] = np.cumsum(dgc[::-1])[::-1]
        dQ[sl], dK[sl], dB[sl] = dQc, dKc, dbeta
        dS = dSp
    return dQ[:L], dK[:L], dV[:L], dB[:L], dLG[:L], dS
