"""Helpers shared by the GPU parity tests: run the CUDA path through the C-ABI
binding and the CPU oracle on the same seeded inputs, and compare.

Tolerances (relative L2 over the whole tensor, float64): 1e-4 for float32
I/O and 2e-2 for bfloat16 I/O, on both the outputs and the final state.  An
element-wise bound is checked too: no element may be off by more than a
fixed fraction of the tensor's RMS (1e-3 for float32, 0.15 for bfloat16),
which catches a few wrong rows that a global norm would average away.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import weight_rnn_gb300 as wr
from weight_rnn_gb300 import synth

TOL_REL = {"f32": 1e-4, "bf16": 2e-2}
TOL_ELEM = {"f32": 1e-3, "bf16": 0.15}


def to_np(t):
    return None if t is None else t.detach().to("cpu", torch.float32).numpy()


def gpu_fwd(inp, w: synth.Workload, device="cuda", h0_gpu=None, chunk=None):
    dev = torch.device(device)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    beta = inp["beta"].to(dev)
    g = None if inp["g"] is None else inp["g"].to(dev)
    h0 = h0_gpu if h0_gpu is not None else (
        None if inp["h0"] is None else inp["h0"].to(dev))
    out, hT = wr.delta_fwd(q, k, v, beta, g, h0, n_h=w.n_h,
                           chunk=chunk or w.chunk)
    torch.cuda.synchronize(dev)
    wr.delta_check_device()
    return out, hT


def oracle_fwd(inp, w: synth.Workload, heads=None, threads=None):
    """Oracle on all heads, or on the listed (b, h) pairs only (each head is
    an independent sequence, so a subset is exact, not an approximation)."""
    q, k, v, beta, g, h0 = (to_np(inp[n]) for n in ("q", "k", "v", "beta", "g", "h0"))
    if heads is None:
        return oracle.fwd(q, k, v, beta, g, h0, n_h=w.n_h, threads=threads)
    outs, states = [], []
    for (b, h) in heads:
        o, s = oracle.fwd(q[b:b + 1, :, h:h + 1], k[b:b + 1, :, :, h:h + 1],
                          v[b:b + 1, :, :, h:h + 1], beta[b:b + 1, :, :, h:h + 1],
                          None if g is None else g[b:b + 1, :, h:h + 1],
                          None if h0 is None else h0[b:b + 1, h:h + 1],
                          n_h=w.n_h, threads=threads)
        outs.append(o[0, :, 0])
        states.append(s[0, 0])
    return np.stack(outs), np.stack(states)


def compare(x, ref, dtype, what):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert x.shape == ref.shape, (what, x.shape, ref.shape)
    assert np.isfinite(x).all(), f"{what}: non-finite values"
    rel = oracle.rel_l2(x, ref)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    worst = float(np.abs(x - ref).max()) / rms if ref.size and rms > 0 else 0.0
    assert rel <= TOL_REL[dtype], f"{what}: rel-L2 {rel:.3e} > {TOL_REL[dtype]:.0e}"
    assert worst <= TOL_ELEM[dtype], (
        f"{what}: max |err| / rms = {worst:.3e} > {TOL_ELEM[dtype]}")
    return rel


def check_full(inp, w, out, hT):
    """Element-by-element against the oracle over every head."""
    ro, rs = oracle_fwd(inp, w)
    e_o = compare(to_np(out), ro, w.dtype, "out")
    e_s = compare(to_np(hT), rs, w.dtype, "hT")
    return e_o, e_s


def check_sampled(inp, w, out, hT, heads):
    """Against the oracle on a sample of heads (full-size workloads)."""
    ro, rs = oracle_fwd(inp, w, heads=heads, threads=len(heads))
    go = to_np(out)
    gs = to_np(hT)
    go = np.stack([go[b, :, h] for (b, h) in heads])
    gs = np.stack([gs[b, h] for (b, h) in heads])
    e_o = compare(go, ro, w.dtype, "out (sampled heads)")
    e_s = compare(gs, rs, w.dtype, "hT (sampled heads)")
    return e_o, e_s
