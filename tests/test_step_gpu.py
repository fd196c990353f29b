"""GPU parity of delta_step (decode, through the C ABI) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import weight_rnn_gb300 as wr
from weight_rnn_gb300 import synth
from parity import compare, to_np

pytestmark = pytest.mark.gpu


def run_steps(w, calls, heads=None, state0=None):
    """Run `calls` decode steps on the GPU; replay the sampled heads (or all)
    through the oracle as one sequence of `calls` tokens from the same start
    state (continuation: successive steps == one forward over the tokens)."""
    dev = torch.device("cuda")
    B, H, dk, dv, n_h = w.B, w.H, w.dk, w.dv, w.n_h
    state = (torch.zeros(B, H, dk, dv, device=dev) if state0 is None
             else state0.to(dev).clone())
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    keep = {n: [] for n in ("q", "k", "v", "beta", "g")}
    outs = []
    bi = torch.tensor([b for b, _ in heads])
    hi = torch.tensor([h for _, h in heads])
    for c in range(calls):
        inp = synth.step_inputs(w, c)
        o = wr.delta_step(*(None if inp[n] is None else inp[n].to(dev)
                            for n in ("q", "k", "v", "beta", "g")), state, n_h=n_h)
        outs.append(o[bi, hi].float().cpu())
        keep["q"].append(inp["q"][bi, hi])
        keep["k"].append(inp["k"][bi, :, hi])
        keep["v"].append(inp["v"][bi, :, hi])
        keep["beta"].append(inp["beta"][bi, :, hi])
        if inp["g"] is not None:
            keep["g"].append(inp["g"][bi, hi])
    torch.cuda.synchronize()
    nH = len(heads)
    # oracle layout: one "batch row" per sampled head, H = 1, T = calls
    q = torch.stack(keep["q"], 1).float().numpy().reshape(nH, calls, 1, dk)
    k = torch.stack(keep["k"], 1).float().numpy().reshape(nH, calls, n_h, 1, dk)
    v = torch.stack(keep["v"], 1).float().numpy().reshape(nH, calls, n_h, 1, dv)
    beta = torch.stack(keep["beta"], 1).numpy().reshape(nH, calls, n_h, 1)
    g = (torch.stack(keep["g"], 1).numpy().reshape(nH, calls, 1) if keep["g"] else None)
    h0 = None if state0 is None else state0[bi, hi].numpy().reshape(nH, 1, dk, dv)
    ro, rs = oracle.fwd(q, k, v, beta, g, h0, n_h=n_h)
    go = torch.stack(outs, 1).numpy()
    gs = to_np(state[bi, hi])
    compare(go, ro[:, :, 0], w.dtype, "decode out")
    compare(gs, rs[:, 0], w.dtype, "decode state")
    return state


def small(dtype="f32", B=3, H=2, dk=128, dv=128, n_h=2, gated=True):
    return synth.WORKLOADS[5].with_(name="small", B=B, H=H, dk=dk, dv=dv, n_h=n_h,
                                    dtype=dtype, gated=gated, seed=77)


@pytest.mark.parametrize("n_h", [1, 2, 3, 4])
@pytest.mark.parametrize("gated", [False, True])
def test_step_substeps(n_h, gated):
    run_steps(small(n_h=n_h, gated=gated), calls=20)


@pytest.mark.parametrize("dk", [16, 32, 64, 128])
@pytest.mark.parametrize("dv", [16, 32, 64, 128])
def test_step_head_dims(dk, dv):
    run_steps(small(dk=dk, dv=dv), calls=9)


def test_step_bf16_io():
    run_steps(small(dtype="bf16"), calls=12)


def test_step_nonzero_start_state():
    w = small()
    s0 = torch.randn(w.B, w.H, w.dk, w.dv, generator=torch.Generator().manual_seed(3)) * 0.1
    run_steps(w, calls=5, state0=s0)


def test_prefill_then_decode_matches_forward():
    """delta_fwd over T tokens, then delta_step per token, equals the oracle
    over all tokens (the state is the whole carried context)."""
    dev = torch.device("cuda")
    w = synth.WORKLOADS[2].with_(B=2, H=2, T=70, n_h=2, dtype="f32", gated=True,
                                 seed=123)
    inp = synth.fwd_inputs(w)
    T1 = 50
    sl = lambda x, s: None if x is None else x[:, s].contiguous()
    pre = {n: sl(inp[n], slice(0, T1)) for n in ("q", "k", "v", "beta", "g")}
    _, state = wr.delta_fwd(*(pre[n].to(dev) for n in ("q", "k", "v", "beta", "g")),
                            n_h=w.n_h, chunk=64)
    outs = []
    for t in range(T1, w.T):
        o = wr.delta_step(inp["q"][:, t].contiguous().to(dev),
                          inp["k"][:, t].contiguous().to(dev),
                          inp["v"][:, t].contiguous().to(dev),
                          inp["beta"][:, t].contiguous().to(dev),
                          inp["g"][:, t].contiguous().to(dev), state, n_h=w.n_h)
        outs.append(o.float().cpu())
    torch.cuda.synchronize()
    ro, rs = oracle.fwd(*(to_np(inp[n]) for n in ("q", "k", "v", "beta", "g")), None,
                        n_h=w.n_h)
    compare(torch.stack(outs, 1).numpy(), ro[:, T1:], "f32", "decode out")
    compare(to_np(state), rs, "f32", "state")


def test_full_size_decode_1024_calls():
    """B256 x H32, dk = dv = 128, n_h = 2, gated, 512 MiB state, 1024 calls;
    the oracle replays every head of four batch rows (128 heads) through all
    1024 tokens."""
    w = synth.WORKLOADS[5]
    heads = [(b, h) for b in (0, 97, 200, w.B - 1) for h in range(w.H)]
    run_steps(w, calls=w.calls, heads=heads)
