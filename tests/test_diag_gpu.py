"""GPU parity of the two diagnostics on the outputs -- the effective rank of a
state ("DeltaProduct" §4.6) and the attention map of the fully parallel form
("08 · linear 路线（三）" §2.4 with the §3 gate) -- against the float64 oracle
functions, through the C ABI."""
import numpy as np
import pytest
import torch

import weight_rnn_gb300 as wr
from weight_rnn_gb300 import synth
from oracle import forms, rel_l2

pytestmark = pytest.mark.gpu

ERANK_TOL = 1e-4   # relative, float32 Jacobi against float64 SVD
MAP_TOL = 1e-4     # rel-L2, float32 arithmetic on the same input bits


def _erank_gpu(S):
    return wr.delta_state_erank(torch.from_numpy(S.astype(np.float32)).cuda()).cpu().numpy()


@pytest.mark.parametrize("dk,dv", [(16, 16), (64, 32), (128, 128), (32, 128)])
def test_erank_random_ranks(dk, dv):
    rng = np.random.default_rng(dk * 1000 + dv)
    B, H = 2, 3
    S = np.zeros((B, H, dk, dv), np.float32)
    ranks = [1, 2, 5, min(dk, dv) // 2, min(dk, dv), min(dk, dv)]
    for i, r in enumerate(ranks):
        b, h = divmod(i, H)
        M = rng.standard_normal((dk, r)) @ (rng.standard_normal((r, dv)) * np.linspace(1, 3, r)[:, None])
        S[b, h] = M.astype(np.float32)
    got = _erank_gpu(S)
    for b in range(B):
        for h in range(H):
            want = forms.effective_rank(S[b, h].astype(np.float64))
            assert abs(got[b, h] - want) <= ERANK_TOL * want, (b, h, got[b, h], want)


def test_erank_closed_forms():
    n = 128
    S = np.zeros((1, 4, n, n), np.float32)
    S[0, 0] = np.eye(n)                                   # n equal singular values
    S[0, 1] = np.outer(np.arange(1, n + 1), np.ones(n))   # rank one
    S[0, 2] = 0.0                                         # the definition does not apply
    S[0, 3] = np.diag(np.r_[np.ones(n - 1), 2.0])         # p = 1/(n+1) (n-1 times), 2/(n+1)
    got = _erank_gpu(S)
    p = np.r_[np.full(n - 1, 1.0 / (n + 1)), 2.0 / (n + 1)]
    assert abs(got[0, 0] - n) <= ERANK_TOL * n
    assert abs(got[0, 1] - 1.0) <= ERANK_TOL
    assert got[0, 2] == 0.0
    assert abs(got[0, 3] - np.exp(-np.sum(p * np.log(p)))) <= ERANK_TOL * n


def test_erank_of_forward_states():
    # the states a real forward leaves behind (small gated workload)
    w = synth.WORKLOADS[3].with_(name="erank", B=2, H=4, T=300)
    inp = synth.fwd_inputs(w)
    d = {n: (None if inp[n] is None else inp[n].cuda()) for n in inp}
    _, hT = wr.delta_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    got = wr.delta_state_erank(hT).cpu().numpy()
    S = hT.cpu().numpy().astype(np.float64)
    for b in range(w.B):
        for h in range(w.H):
            want = forms.effective_rank(S[b, h])
            assert abs(got[b, h] - want) <= ERANK_TOL * want


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("N,dk", [(1, 16), (17, 128), (64, 128), (64, 32)])
def test_attention_map(dtype, gated, N, dk):
    w = synth.WORKLOADS[2].with_(name="map", B=2, H=3, T=N, dk=dk, dv=dk, dtype=dtype,
                                 gated=gated, h0_std=0.0, seed=N * 7 + dk)
    inp = synth.fwd_inputs(w)
    q, k = inp["q"], inp["k"].reshape(w.B, N, w.H, dk)
    beta = inp["beta"].reshape(w.B, N, w.H)
    g = inp["g"]
    attn = wr.delta_attention_map(q.cuda(), k.cuda(), beta.cuda(),
                                  None if g is None else g.cuda()).cpu().numpy()
    qf, kf, bf = (x.to(torch.float64).numpy() for x in (q, k, beta))
    lg = None if g is None else np.log(g.to(torch.float64).numpy())
    for b in range(w.B):
        for h in range(w.H):
            want = forms.attention_map(qf[b, :, h], kf[b, :, h], bf[b, :, h],
                                       None if lg is None else lg[b, :, h])
            assert rel_l2(attn[b, h], want) <= MAP_TOL, (b, h)
            assert np.all(np.triu(attn[b, h], 1) == 0.0)
