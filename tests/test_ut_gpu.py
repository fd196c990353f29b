"""GPU parity of the intra-chunk pass (delta_ut_transform, through the C ABI)
against the oracle's UT transform ("08 · linear 路线（三）" §2.2 with the §3
gate), and of the two-pass forward (delta_ut_transform, then
delta_fwd_with_ut) against delta_fwd and the oracle."""
import numpy as np
import pytest
import torch

import oracle
import weight_rnn_gb300 as wr
from oracle import forms
from weight_rnn_gb300 import synth
from parity import check_full, gpu_fwd, to_np

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


def small(B=2, H=3, T=200, n_h=1, gated=True, beta_scale=1.0, seed=7):
    return W[2].with_(name="small", B=B, H=H, T=T, n_h=n_h, gated=gated,
                      h0_std=0.05 if gated else 0.0, beta_scale=beta_scale, seed=seed)


def oracle_t(inp, w, C=64):
    """T of every chunk of every head, float64, from the oracle's UT form on
    the extended sequence ("DeltaProduct" §4.1).  A gate of exactly 0 enters
    as log g = -1e4 (exp underflows to 0 in float64; the kernels clamp log g
    at -80, exp(-80) ~ 2e-35)."""
    k = to_np(inp["k"]).reshape(w.B, w.T, w.n_h, w.H, w.dk)
    beta = to_np(inp["beta"]).reshape(w.B, w.T, w.n_h, w.H)
    g = None if inp["g"] is None else to_np(inp["g"]).astype(np.float64)
    L = w.T * w.n_h
    nt = -(-L // C)
    out = np.zeros((w.B, w.H, nt, C, C))
    for b in range(w.B):
        for h in range(w.H):
            lg = None
            if g is not None:
                lg = np.zeros(L)
                gv = g[b, :, h]
                lg[0::w.n_h] = np.where(gv > 0, np.log(np.maximum(gv, 1e-300)), -1e4)
            out[b, h] = forms.ut_transform(k[b, :, :, h].reshape(L, w.dk).astype(np.float64),
                                           beta[b, :, :, h].reshape(L), lg, C)
    return out


def gpu_t(inp, w):
    dev = torch.device("cuda")
    k = inp["k"].to(dev)
    beta = inp["beta"].to(dev)
    g = None if inp["g"] is None else inp["g"].to(dev)
    t = wr.delta_ut_transform(k, beta, g, n_h=w.n_h, chunk=64)
    torch.cuda.synchronize()
    wr.delta_check_device()
    return t


def compare_t(x, ref, what="T"):
    """T against the oracle: the global relative L2 bound of every bf16
    comparison (2e-2), and per chunk no entry off by more than 2e-2 of the
    chunk's largest entry.  The entries are rounded to bf16 (relative 2^-9)
    after a float32 solve whose block merges run on tf32 inputs (2^-11), and
    many entries are exactly 0, so a bound relative to the RMS of the whole
    tensor would be meaningless here."""
    x = np.asarray(x, np.float64)
    assert x.shape == ref.shape, (what, x.shape, ref.shape)
    assert np.isfinite(x).all(), f"{what}: non-finite values"
    rel = oracle.rel_l2(x, ref)
    assert rel <= 2e-2, f"{what}: rel-L2 {rel:.3e} > 2e-2"
    err = np.abs(x - ref).reshape(-1, ref.shape[-2] * ref.shape[-1]).max(axis=1)
    scale = np.abs(ref).reshape(-1, ref.shape[-2] * ref.shape[-1]).max(axis=1)
    bad = err > 2e-2 * scale + 1e-30
    assert not bad.any(), (f"{what}: {int(bad.sum())} chunks with max |err| > 2e-2 max |T|, "
                           f"worst {float((err / np.maximum(scale, 1e-30)).max()):.3e}")
    return rel


def check_t(inp, w):
    t = gpu_t(inp, w)
    ref = oracle_t(inp, w)
    compare_t(to_np(t), ref)
    # identity steps past the end of the sequence: zero rows and columns
    L = w.T * w.n_h
    r = L - 64 * (ref.shape[2] - 1)
    if r < 64:
        last = to_np(t)[:, :, -1]
        assert not last[:, :, r:].any() and not last[:, :, :, r:].any()
    return t


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("T", [1, 64, 130, 200])
def test_ut_transform(gated, T):
    check_t(synth.fwd_inputs(small(T=T, gated=gated, seed=T)), small(T=T, gated=gated, seed=T))


def test_ut_transform_odd_chunk_count():
    """An odd number of chunks over all heads: the last pair of the pass has
    one chunk only."""
    w = small(B=1, H=3, T=130, seed=3)
    check_t(synth.fwd_inputs(w), w)


@pytest.mark.parametrize("n_h", [2, 3, 4])
def test_ut_transform_deltaproduct(n_h):
    w = small(T=97, n_h=n_h, beta_scale=2.0, seed=40 + n_h)
    check_t(synth.fwd_inputs(w), w)


def test_ut_transform_beta_extremes_and_resets():
    w = small(T=160, n_h=2, beta_scale=2.0, seed=99)
    inp = synth.fwd_inputs(w)
    inp["beta"][:, 10:20] = 0.0
    inp["beta"][:, 40:50] = 2.0
    inp["g"][:, [5, 64, 65, 127, 159]] = 0.0
    check_t(inp, w)


def test_ut_transform_many_chunks_per_cta():
    """More chunk pairs than resident CTAs: every CTA loops over several
    pairs and reuses both of its slots; checked on a sample of heads."""
    w = small(B=4, H=40, T=1000, seed=5)
    inp = synth.fwd_inputs(w)
    t = gpu_t(inp, w)
    for (b, h) in [(0, 0), (1, 17), (3, 39)]:
        one = dict(k=inp["k"][b:b + 1, :, :, h:h + 1].contiguous(),
                   beta=inp["beta"][b:b + 1, :, :, h:h + 1].contiguous(),
                   g=inp["g"][b:b + 1, :, h:h + 1].contiguous())
        compare_t(to_np(t[b:b + 1, h:h + 1]), oracle_t(one, w.with_(B=1, H=1)), f"T head {(b, h)}")


@pytest.mark.parametrize("gated,n_h", [(False, 1), (True, 1), (True, 3)])
def test_two_passes_equal_delta_fwd(gated, n_h):
    """delta_ut_transform + delta_fwd_with_ut (caller-held T) give the same
    bits as delta_fwd (library scratch), and match the oracle."""
    w = small(B=2, H=5, T=333, gated=gated, n_h=n_h, seed=17 + n_h)
    inp = synth.fwd_inputs(w)
    dev = torch.device("cuda")
    d = {n: (None if inp[n] is None else inp[n].to(dev)) for n in inp}
    t = wr.delta_ut_transform(d["k"], d["beta"], d["g"], n_h=n_h)
    o2, s2 = wr.delta_fwd_with_ut(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], t,
                                  n_h=n_h)
    o1, s1 = gpu_fwd(inp, w)
    torch.cuda.synchronize()
    check_full(inp, w, o2, s2)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    # the UT pass again, now on shared memory the state pass has used: the
    # same bits (nothing it reads is left over from an earlier kernel)
    t2 = wr.delta_ut_transform(d["k"], d["beta"], d["g"], n_h=n_h)
    torch.cuda.synchronize()
    assert torch.equal(t, t2)
