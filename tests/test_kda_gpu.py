"""GPU parity of the channel-wise-gate (KDA) entry points (delta_fwd_kda,
delta_step_kda; the KDA row of "08 · linear 路线（三）" §1.4) against the
oracle's float64 recurrence ``oracle.forms.kda_recurrent``, head by head."""
import numpy as np
import pytest
import torch

from oracle import forms
import weight_rnn_gb300 as wr
from parity import compare, to_np

pytestmark = pytest.mark.gpu


def kda_inputs(B, T, H, dk, dv, n_h, dtype, h0, seed):
    gen = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=gen)
    k = r(B, T, n_h, H, dk)
    k = k / k.norm(dim=-1, keepdim=True)
    return {
        "q": r(B, T, H, dk).to(dtype),
        "k": k.to(dtype),
        "v": r(B, T, n_h, H, dv).to(dtype),
        "beta": torch.sigmoid(r(B, T, n_h, H)) * (2.0 if n_h > 1 else 1.0),
        # per-channel gates from near 1 down to resets
        "alpha": torch.sigmoid(r(B, T, H, dk) * 2.0 + 2.5),
        "h0": r(B, H, dk, dv) * 0.1 if h0 else None,
    }


def oracle_kda(inp, n_h):
    q, k, v, beta, alpha, h0 = (to_np(inp[n]) for n in ("q", "k", "v", "beta", "alpha", "h0"))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, T, H, dv))
    hT = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            o, S = forms.kda_recurrent(q[b, :, h], k[b, :, :, h], v[b, :, :, h], beta[b, :, :, h],
                                       alpha[b, :, h], None if h0 is None else h0[b, h], n_h=n_h)
            out[b, :, h] = o
            hT[b, h] = S
    return out, hT


@pytest.mark.parametrize("dtype,dk,dv,n_h,chunk,T,h0", [
    (torch.float32, 32, 16, 1, 16, 70, True),
    (torch.float32, 16, 32, 2, 32, 45, False),
    (torch.float32, 64, 64, 1, 64, 130, True),
    (torch.bfloat16, 128, 128, 1, 64, 100, True),   # the tensor-core shape takes the CUDA-core kernel
    (torch.bfloat16, 64, 32, 3, 16, 33, False),
])
def test_fwd_kda_matches_oracle(dtype, dk, dv, n_h, chunk, T, h0):
    B, H = 2, 2
    inp = kda_inputs(B, T, H, dk, dv, n_h, dtype, h0, seed=dk * 13 + T)
    inp["alpha"][0, 5, 1, :dk // 2] = 0.0  # half the channels reset at one step
    dev = torch.device("cuda")
    d = {n: None if inp[n] is None else inp[n].to(dev) for n in inp}
    out, hT = wr.delta_fwd_kda(d["q"], d["k"], d["v"], d["beta"], d["alpha"], d["h0"],
                               n_h=n_h, chunk=chunk)
    torch.cuda.synchronize()
    ro, rs = oracle_kda(inp, n_h)
    tol = "bf16" if dtype == torch.bfloat16 else "f32"
    compare(to_np(out), ro, tol, "out")
    compare(to_np(hT), rs, tol, "hT")


def test_fwd_kda_with_channel_constant_gate_equals_delta_fwd():
    # alpha equal on every channel is Gated DeltaNet: the same result as
    # delta_fwd's scalar gate on the CUDA-core kernel (float32)
    B, T, H, dk, dv = 2, 50, 2, 32, 32
    inp = kda_inputs(B, T, H, dk, dv, 1, torch.float32, True, seed=5)
    g = inp["alpha"][..., 0].contiguous()
    inp["alpha"] = g[..., None].expand(B, T, H, dk).contiguous()
    dev = torch.device("cuda")
    d = {n: None if inp[n] is None else inp[n].to(dev) for n in inp}
    o1, s1 = wr.delta_fwd_kda(d["q"], d["k"], d["v"], d["beta"], d["alpha"], d["h0"], chunk=16)
    o2, s2 = wr.delta_fwd(d["q"], d["k"], d["v"], d["beta"], g.to(dev), d["h0"], chunk=16)
    torch.cuda.synchronize()
    compare(to_np(o1), to_np(o2), "f32", "out")
    compare(to_np(s1), to_np(s2), "f32", "hT")


@pytest.mark.parametrize("dtype,dk,dv,n_h", [(torch.float32, 128, 128, 2),
                                             (torch.bfloat16, 64, 64, 1),
                                             (torch.float32, 32, 16, 3)])
def test_step_kda_matches_oracle_over_calls(dtype, dk, dv, n_h):
    B, H, calls = 2, 3, 4
    dev = torch.device("cuda")
    gen = torch.Generator().manual_seed(dk + n_h)
    state = torch.zeros(B, H, dk, dv, device=dev)
    ref = [[None] * H for _ in range(B)]
    for c in range(calls):
        inp = kda_inputs(B, 1, H, dk, dv, n_h, dtype, False, seed=1000 + c * 7 + dk)
        q, k, v = inp["q"][:, 0], inp["k"][:, 0], inp["v"][:, 0]
        beta, alpha = inp["beta"][:, 0], inp["alpha"][:, 0]
        out = wr.delta_step_kda(q.to(dev), k.to(dev), v.to(dev), beta.to(dev), alpha.to(dev),
                                state, n_h=n_h)
        torch.cuda.synchronize()
        ro = np.zeros((B, H, dv))
        for b in range(B):
            for h in range(H):
                o, S = forms.kda_recurrent(to_np(q[b, h])[None], to_np(k[b, :, h])[None],
                                           to_np(v[b, :, h])[None], to_np(beta[b, :, h])[None],
                                           to_np(alpha[b, h])[None], ref[b][h], n_h=n_h)
                ro[b, h] = o[0]
                ref[b][h] = S
        tol = "bf16" if dtype == torch.bfloat16 else "f32"
        compare(to_np(out), ro, tol, f"out of call {c}")
    compare(to_np(state), np.array(ref), "bf16" if dtype == torch.bfloat16 else "f32", "state")
