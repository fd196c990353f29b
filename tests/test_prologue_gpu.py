"""GPU parity of the input prologue entry points (delta_fwd_prologue,
delta_step_prologue; "DeltaProduct" §2.2, the query path of the layer design
in "08 · linear 路线（三）" §3) against the oracle's float64 prologue followed
by the float64 recurrence, on raw seeded projections."""
import numpy as np
import pytest
import torch

import oracle
from oracle import forms
import weight_rnn_gb300 as wr
from parity import compare, to_np

pytestmark = pytest.mark.gpu


def raw_inputs(B, T, H, dk, dv, n_h, dtype, gated, h0, seed):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=gen)
    inp = {
        "q": r(B, T, H, dk).to(dtype),
        "k": r(B, T, n_h, H, dk).to(dtype) * 1.5,
        "v": r(B, T, n_h, H, dv).to(dtype),
        "beta": r(B, T, n_h, H) * 2.0,
        "g": torch.sigmoid(r(B, T, H) * 2.0 + 3.0) if gated else None,
        "h0": r(B, H, dk, dv) * 0.05 if h0 else None,
    }
    return inp


def oracle_prologue_fwd(inp, n_h, beta_map):
    q, k, b = forms.prologue(to_np(inp["q"]), to_np(inp["k"]), to_np(inp["beta"]), beta_map)
    return oracle.fwd(q, k, to_np(inp["v"]), b, to_np(inp["g"]), to_np(inp["h0"]), n_h=n_h)


CASES = [
    # the tensor-core path (bf16, d = 128, chunk 64)
    dict(B=2, T=200, H=3, dk=128, dv=128, n_h=1, chunk=64, dtype=torch.bfloat16, gated=True, h0=True),
    dict(B=1, T=130, H=2, dk=128, dv=128, n_h=3, chunk=64, dtype=torch.bfloat16, gated=True, h0=False),
    dict(B=2, T=97, H=2, dk=128, dv=128, n_h=1, chunk=64, dtype=torch.bfloat16, gated=False, h0=False),
    # the CUDA-core path (float32 I/O, small heads)
    dict(B=2, T=50, H=2, dk=32, dv=16, n_h=2, chunk=16, dtype=torch.float32, gated=True, h0=True),
    dict(B=1, T=33, H=3, dk=16, dv=32, n_h=1, chunk=32, dtype=torch.float32, gated=False, h0=False),
]


@pytest.mark.parametrize("beta_map", ["sigmoid", "2sigmoid"])
@pytest.mark.parametrize("c", CASES, ids=lambda c: f"{c['dtype']}-d{c['dk']}x{c['dv']}-nh{c['n_h']}-T{c['T']}")
def test_fwd_prologue_matches_oracle(c, beta_map):
    inp = raw_inputs(c["B"], c["T"], c["H"], c["dk"], c["dv"], c["n_h"], c["dtype"], c["gated"],
                     c["h0"], seed=c["T"] * 7 + c["dk"])
    # a zero key row: its SiLU is zero, so that sub-step leaves the state alone
    inp["k"][0, 3, 0, 0] = 0
    dev = torch.device("cuda")
    d = {n: None if inp[n] is None else inp[n].to(dev) for n in inp}
    out, hT = wr.delta_fwd_prologue(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                    n_h=c["n_h"], chunk=c["chunk"], beta_map=beta_map)
    torch.cuda.synchronize()
    wr.delta_check_device()
    ro, rs = oracle_prologue_fwd(inp, c["n_h"], beta_map)
    tol = "bf16" if c["dtype"] == torch.bfloat16 else "f32"
    compare(to_np(out), ro, tol, "out")
    compare(to_np(hT), rs, tol, "hT")


def test_fwd_prologue_empty_sequence_copies_the_state():
    dev = torch.device("cuda")
    h0 = torch.randn(1, 2, 128, 128, device=dev)
    z = lambda *s: torch.zeros(*s, device=dev, dtype=torch.bfloat16)
    out, hT = wr.delta_fwd_prologue(z(1, 0, 2, 128), z(1, 0, 2, 128), z(1, 0, 2, 128),
                                    torch.zeros(1, 0, 2, device=dev), None, h0)
    torch.cuda.synchronize()
    assert out.numel() == 0 and torch.equal(hT, h0)


@pytest.mark.parametrize("dtype,dk,dv,n_h,beta_map", [
    (torch.float32, 128, 128, 2, "2sigmoid"),
    (torch.bfloat16, 128, 128, 1, "sigmoid"),
    (torch.float32, 32, 64, 3, "sigmoid"),
])
def test_step_prologue_matches_oracle_over_calls(dtype, dk, dv, n_h, beta_map):
    B, H, calls = 3, 4, 5
    dev = torch.device("cuda")
    gen = torch.Generator().manual_seed(dk * 31 + n_h)
    state = torch.zeros(B, H, dk, dv, device=dev)
    ref = None
    for c in range(calls):
        q = torch.randn(B, H, dk, generator=gen).to(dtype)
        k = torch.randn(B, n_h, H, dk, generator=gen).to(dtype)
        v = torch.randn(B, n_h, H, dv, generator=gen).to(dtype)
        b = torch.randn(B, n_h, H, generator=gen) * 2.0
        g = torch.sigmoid(torch.randn(B, H, generator=gen) + 3.0)
        if c == 1:
            k[1, 0, 2] = 0  # a zero key: an identity sub-step
        out = wr.delta_step_prologue(q.to(dev), k.to(dev), v.to(dev), b.to(dev), g.to(dev), state,
                                     n_h=n_h, beta_map=beta_map)
        torch.cuda.synchronize()
        qn, kn, bn = forms.prologue(to_np(q), to_np(k), to_np(b), beta_map)
        ro, ref = oracle.step(qn, kn, to_np(v), bn, to_np(g), ref, n_h=n_h)
        tol = "bf16" if dtype == torch.bfloat16 else "f32"
        compare(to_np(out), ro, tol, f"out of call {c}")
    compare(to_np(state), ref, "bf16" if dtype == torch.bfloat16 else "f32", "state")


@pytest.mark.parametrize("dtype,dk,n_h", [(torch.bfloat16, 128, 1), (torch.bfloat16, 64, 3),
                                          (torch.float32, 128, 2), (torch.float32, 16, 1)])
def test_prologue_alone_matches_oracle(dtype, dk, n_h):
    B, T, H = 2, 37, 3
    gen = torch.Generator().manual_seed(dk + n_h)
    q = (torch.randn(B, T, H, dk, generator=gen) * 3).to(dtype)
    k = (torch.randn(B, T, n_h, H, dk, generator=gen) * 3).to(dtype)
    b = torch.randn(B, T, n_h, H, generator=gen) * 4
    q[0, 0, 0] = 0  # a zero row stays zero
    dev = torch.device("cuda")
    for beta_map in ("sigmoid", "2sigmoid"):
        qo, ko, bo = wr.delta_prologue(q.to(dev), k.to(dev), b.to(dev), n_h=n_h, beta_map=beta_map)
        torch.cuda.synchronize()
        rq, rk, rb = forms.prologue(to_np(q), to_np(k), to_np(b), beta_map)
        # float32 arithmetic, then rounding to the I/O type
        atol = 4e-3 if dtype == torch.bfloat16 else 2e-6
        np.testing.assert_allclose(to_np(qo), rq, rtol=0, atol=atol)
        np.testing.assert_allclose(to_np(ko), rk, rtol=0, atol=atol)
        np.testing.assert_allclose(to_np(bo), rb, rtol=1e-5, atol=0)  # __expf: a few ulp
        assert torch.all(qo[0, 0, 0] == 0)
        np.testing.assert_allclose(np.linalg.norm(to_np(ko), axis=-1), 1.0, atol=8 * atol)
