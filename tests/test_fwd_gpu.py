"""GPU parity of delta_fwd (through the C ABI) against the float64 CPU oracle."""
import numpy as np
import pytest
import torch

import weight_rnn_gb300 as wr
from weight_rnn_gb300 import synth
from parity import check_full, check_sampled, compare, gpu_fwd, oracle_fwd, to_np

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


def small(dtype="bf16", B=2, H=3, T=200, dk=128, dv=128, n_h=1, chunk=64,
          gated=True, h0=0.05, beta_scale=1.0, seed=7):
    return W[2].with_(name="small", B=B, H=H, T=T, dk=dk, dv=dv, n_h=n_h, chunk=chunk,
                      dtype=dtype, gated=gated, h0_std=h0, beta_scale=beta_scale,
                      seed=seed)


def run_full(w):
    inp = synth.fwd_inputs(w)
    out, hT = gpu_fwd(inp, w)
    return check_full(inp, w, out, hT)


def test_workload1_smoke_f32():
    """B1 H1 T64 d16 float32 chunk 16 -- every element against the oracle."""
    run_full(W[1])


# --- the tensor-core shape (bf16, d = 128, chunk 64), ragged lengths --------
@pytest.mark.parametrize("T", [1, 63, 64, 65, 130, 1000])
@pytest.mark.parametrize("gated,h0", [(False, 0.0), (True, 0.05)])
def test_bf16_d128_c64_lengths(T, gated, h0):
    run_full(small(T=T, gated=gated, h0=h0, seed=T))


@pytest.mark.parametrize("n_h", [1, 2, 3, 4])
def test_deltaproduct_substeps(n_h):
    # T * n_h is not a multiple of 64 for n_h = 3: token groups straddle chunks
    run_full(small(T=97, n_h=n_h, beta_scale=2.0, seed=30 + n_h))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk", [16, 32, 64, 128])
@pytest.mark.parametrize("dv", [16, 32, 64, 128])
def test_head_dims(dtype, dk, dv):
    run_full(small(dtype=dtype, dk=dk, dv=dv, T=75, chunk=32, n_h=2, seed=dk + dv))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_chunk_sizes(dtype, chunk):
    run_full(small(dtype=dtype, chunk=chunk, T=150, seed=chunk))


def test_beta_extremes_and_resets():
    """beta in {0, 1, 2} (identity step, projection, reflection) and g = 0
    (a reset, log g clamped inside the kernels)."""
    w = small(T=160, n_h=2, beta_scale=2.0, seed=99)
    inp = synth.fwd_inputs(w)
    beta = inp["beta"]
    beta[:, 10:20] = 0.0
    beta[:, 40:50] = 1.0
    beta[:, 70:80] = 2.0
    g = inp["g"]
    g[:, [5, 64, 65, 127, 159]] = 0.0
    out, hT = gpu_fwd(inp, w)
    check_full(inp, w, out, hT)


def test_empty_sequence_passes_state_through():
    w = small(T=0)
    inp = synth.fwd_inputs(w)
    out, hT = gpu_fwd(inp, w)
    assert out.numel() == 0
    assert torch.equal(hT.cpu(), inp["h0"])
    w0 = small(T=0, h0=0.0)
    out, hT = gpu_fwd(synth.fwd_inputs(w0), w0)
    assert torch.count_nonzero(hT) == 0


def test_empty_batch():
    w = small(B=0)
    inp = synth.fwd_inputs(w)
    out, hT = gpu_fwd(inp, w)
    assert out.numel() == 0 and hT.numel() == 0


def test_state_in_place_and_continuation():
    """hT may alias h0; running T1 then T2 tokens from the carried state
    equals running T1 + T2 tokens at once (checked against the oracle)."""
    w = small(T=300, n_h=2, seed=5)
    inp = synth.fwd_inputs(w)
    dev = torch.device("cuda")
    T1 = 173
    part = lambda x, s: None if x is None else x[:, s].contiguous()
    state = inp["h0"].to(dev).clone()
    outs = []
    for s in (slice(0, T1), slice(T1, None)):
        sub = dict(q=part(inp["q"], s), k=part(inp["k"], s), v=part(inp["v"], s),
                   beta=part(inp["beta"], s), g=part(inp["g"], s), h0=None)
        o, hT = wr.delta_fwd(*(sub[n].to(dev) for n in ("q", "k", "v", "beta", "g")),
                             state, None, state, n_h=w.n_h, chunk=w.chunk)
        assert hT.data_ptr() == state.data_ptr()
        outs.append(o)
    torch.cuda.synchronize()
    ro, rs = oracle_fwd(inp, w)
    compare(to_np(torch.cat(outs, 1)), ro, w.dtype, "out")
    compare(to_np(state), rs, w.dtype, "hT")


def test_deterministic():
    w = small(T=500, n_h=3, seed=11)
    inp = synth.fwd_inputs(w)
    o1, s1 = gpu_fwd(inp, w)
    o2, s2 = gpu_fwd(inp, w)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("gated,n_h", [(False, 1), (True, 1), (True, 3)])
def test_repeated_launches_are_bitwise_identical(gated, n_h):
    """The tensor-core kernel hands every intermediate between warp roles
    through barriers; a missing wait shows up as run-to-run differences.
    Many heads (one CTA each) and many chunks, several launches, bitwise."""
    w = small(B=4, H=16, T=1024, gated=gated, n_h=n_h, h0=0.05 if gated else 0.0,
              seed=123 + n_h)
    inp = synth.fwd_inputs(w)
    o0, s0 = gpu_fwd(inp, w)
    for _ in range(4):
        o, s_ = gpu_fwd(inp, w)
        assert torch.equal(o, o0) and torch.equal(s_, s0)
    heads = [(0, 0), (1, 7), (3, 15)]
    check_sampled(inp, w, o0, s0, heads)


def test_misaligned_pointer_is_rejected():
    w = small(T=8)
    inp = synth.fwd_inputs(w)
    dev = torch.device("cuda")
    q = torch.empty(inp["q"].numel() + 1, dtype=inp["q"].dtype, device=dev)[1:]
    q = q.view(inp["q"].shape)
    with pytest.raises(wr.DeltaError) as ei:
        wr.delta_fwd(q, inp["k"].to(dev), inp["v"].to(dev), inp["beta"].to(dev),
                     n_h=1, chunk=64)
    assert ei.value.status == wr.DELTA_ERR_ALIGN


# --- full-size workloads, in the launch configuration the bench times --------
@pytest.mark.parametrize("wid", [2, 3, 4])
def test_full_size_workload(wid):
    """Every head of the full-size workload against the oracle (threaded over
    the host cores), element by element."""
    w = W[wid]
    inp = synth.fwd_inputs(w)
    out, hT = gpu_fwd(inp, w)
    assert out.shape == (w.B, w.T, w.H, w.dv) and hT.shape == (w.B, w.H, w.dk, w.dv)
    check_full(inp, w, out, hT)
