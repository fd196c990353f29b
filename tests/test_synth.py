"""The seeded input recipe on CPU: the shapes, layouts and value ranges each
workload's inputs are documented to have, and that a seed fixes them."""
import torch

from weight_rnn_gb300 import synth


def small(wid, **kw):
    w = synth.WORKLOADS[wid]
    return w.with_(**{"B": 1, "H": 2, "T": min(w.T, 33), **kw})


def test_forward_inputs_follow_the_recipe():
    for wid in (1, 2, 3, 4):
        w = small(wid)
        x = synth.fwd_inputs(w)
        B, T, H, n_h, dk, dv = w.B, w.T, w.H, w.n_h, w.dk, w.dv
        assert x["q"].shape == (B, T, H, dk) and x["k"].shape == (B, T, n_h, H, dk)
        assert x["v"].shape == (B, T, n_h, H, dv) and x["beta"].shape == (B, T, n_h, H)
        assert x["q"].dtype == synth.torch_dtype(w.dtype) == x["k"].dtype == x["v"].dtype
        # unit queries and keys (to the I/O dtype's rounding)
        tol = 1e-2 if w.dtype == "bf16" else 1e-5
        for n in ("q", "k"):
            norms = x[n].float().norm(dim=-1)
            assert torch.allclose(norms, torch.ones_like(norms), atol=tol), (wid, n)
        # beta in (0, beta_scale); the gate in (0, 1]; h0 only where given
        assert float(x["beta"].min()) > 0 and float(x["beta"].max()) < w.beta_scale
        if w.gated:
            assert x["g"].shape == (B, T, H)
            assert float(x["g"].min()) > 0 and float(x["g"].max()) <= 1
        else:
            assert x["g"] is None
        assert (x["h0"] is None) == (w.h0_std == 0)


def test_silu_keys_lean_positive_and_the_initial_state_has_its_spread():
    w = small(3, H=4, T=64)
    x = synth.fwd_inputs(w)
    # E[SiLU(N)] ~ 0.21 and E[SiLU(N)^2] ~ 0.36: a normalised 128-vector of
    # them has mean entry ~ 0.21 / sqrt(128 * 0.36) ~ 0.03, and the negative
    # entries are small (SiLU >= -0.28); plain L2(N(0,1)) keys average ~ 0
    k = x["k"].float()
    assert float(k.mean()) > 0.02
    assert float(synth.fwd_inputs(small(1))["k"].float().mean().abs()) < 0.05
    assert abs(float(x["h0"].std()) - w.h0_std) < 0.1 * w.h0_std


def test_a_seed_fixes_the_inputs_and_decode_calls_differ():
    w = small(2)
    a, b = synth.fwd_inputs(w), synth.fwd_inputs(w)
    assert all(torch.equal(a[n], b[n]) for n in ("q", "k", "v", "beta"))
    c = synth.fwd_inputs(w, seed=w.seed + 1)
    assert not torch.equal(a["v"], c["v"])
    d = synth.WORKLOADS[5].with_(B=2, H=2)
    s0, s1 = synth.step_inputs(d, 0), synth.step_inputs(d, 1)
    assert s0["q"].shape == (2, 2, 128) and s0["k"].shape == (2, 2, 2, 128)
    assert not torch.equal(s0["k"], s1["k"])
    assert torch.equal(s1["k"], synth.step_inputs(d, 1)["k"])
