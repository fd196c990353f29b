"""GPU parity of delta_bwd (the gradients of delta_fwd; no page states
backward formulas) against the oracle's float64 autograd of the recurrence,
head by head, and a first-order check against delta_fwd itself."""
import numpy as np
import pytest
import torch

from oracle import forms
import weight_rnn_gb300 as wr
from parity import compare, to_np

pytestmark = pytest.mark.gpu


def inputs(B, T, H, dk, dv, n_h, dtype, gated, h0, seed):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=gen)
    k = r(B, T, n_h, H, dk)
    k = k / k.norm(dim=-1, keepdim=True)
    return {
        "q": r(B, T, H, dk).to(dtype), "k": k.to(dtype), "v": r(B, T, n_h, H, dv).to(dtype),
        "beta": torch.sigmoid(r(B, T, n_h, H)) * (2.0 if n_h > 1 else 1.0),
        "g": torch.sigmoid(r(B, T, H) * 2.0 + 2.0) if gated else None,
        "h0": r(B, H, dk, dv) * 0.2 if h0 else None,
        "dout": r(B, T, H, dv).to(dtype), "dhT": r(B, H, dk, dv) * 0.5,
    }


def oracle_grads(inp, n_h):
    q, k, v, beta, g, h0, dout, dhT = (to_np(inp[n]) for n in
                                       ("q", "k", "v", "beta", "g", "h0", "dout", "dhT"))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    res = [np.zeros_like(q, dtype=np.float64), np.zeros((B, T, n_h, H, dk)), np.zeros((B, T, n_h, H, dv)),
           np.zeros((B, T, n_h, H)), None if g is None else np.zeros((B, T, H)), np.zeros((B, H, dk, dv))]
    for b in range(B):
        for h in range(H):
            gq, gk, gv, gb, gg, gs = forms.recurrent_grad(
                q[b, :, h], k[b, :, :, h], v[b, :, :, h], beta[b, :, :, h],
                None if g is None else g[b, :, h], None if h0 is None else h0[b, h],
                dout[b, :, h], dhT[b, h], n_h=n_h)
            res[0][b, :, h], res[1][b, :, :, h], res[2][b, :, :, h] = gq, gk, gv
            res[3][b, :, :, h], res[5][b, h] = gb, gs
            if g is not None:
                res[4][b, :, h] = gg
    return res


@pytest.mark.parametrize("dtype,dk,dv,n_h,T,gated,h0", [
    (torch.float32, 16, 16, 1, 40, True, True),
    (torch.float32, 32, 16, 2, 70, True, False),
    (torch.float32, 64, 32, 3, 25, False, True),
    (torch.float32, 128, 128, 1, 150, True, True),   # more than two blocks of 64 sub-steps
    (torch.float32, 128, 64, 1, 70, True, True),     # two groups of 32 value columns
    (torch.float32, 16, 128, 2, 33, True, False),    # four groups, narrow keys
    (torch.bfloat16, 128, 128, 1, 66, True, True),
])
def test_bwd_matches_oracle(dtype, dk, dv, n_h, T, gated, h0):
    B, H = 2, 2
    inp = inputs(B, T, H, dk, dv, n_h, dtype, gated, h0, seed=dk * 3 + T + n_h)
    if gated:
        inp["g"][0, 10, 1] = 0.0    # a reset: dg still flows, nothing passes it
        if T > 64:
            inp["g"][1, 64, 0] = 0.0  # ... and one at the start of a recomputed block
    dev = torch.device("cuda")
    d = {n: None if inp[n] is None else inp[n].to(dev) for n in inp}
    got = wr.delta_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["dout"], d["dhT"], n_h=n_h)
    torch.cuda.synchronize()
    ref = oracle_grads(inp, n_h)
    names = ("dq", "dk", "dv", "dbeta", "dg", "dh0")
    for name, x, r in zip(names, got, ref):
        if r is None:
            assert x is None
            continue
        # the inputs are exact in float32: the float32 tolerance applies to both I/O types
        compare(to_np(x).reshape(r.shape), r, "f32", name)


def test_bwd_is_the_derivative_of_the_forward():
    # <dout, d out> + <dhT, d hT> for a small step along a random direction
    # equals the directional derivative from the gradients (float32 forward)
    B, T, H, dk, dv = 1, 30, 2, 32, 32
    inp = inputs(B, T, H, dk, dv, 1, torch.float32, True, True, seed=77)
    dev = torch.device("cuda")
    d = {n: None if inp[n] is None else inp[n].to(dev) for n in inp}
    gq, gk, gv, gb, gg, gh = wr.delta_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                          d["dout"], d["dhT"])
    gen = torch.Generator().manual_seed(78)
    dirs = {n: torch.randn(d[n].shape, generator=gen).to(dev) for n in ("q", "k", "v", "h0")}
    eps = 1e-3

    def L(s):
        x = {n: d[n] + s * dirs[n] if n in dirs else d[n] for n in d}
        o, hT = wr.delta_fwd(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], chunk=16)
        return float((o * d["dout"]).sum() + (hT * d["dhT"]).sum())
    fd = (L(eps) - L(-eps)) / (2 * eps)
    an = float(sum((gr * dirs[n]).sum() for n, gr in (("q", gq), ("k", gk), ("v", gv), ("h0", gh))))
    assert abs(fd - an) <= 2e-3 * max(1.0, abs(an)), (fd, an)
