"""Failure detection on the GPU without a fault: a bounded wait that runs out
reports through the device error word and leaves the context usable; an
injected host-side failure reaches the caller and the next call recovers."""
import pytest
import torch

import weight_rnn_gb300 as wr
from weight_rnn_gb300 import synth
from parity import check_full, gpu_fwd

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


def small():
    return W[2].with_(name="small", B=2, H=3, T=130, n_h=2, gated=True, h0_std=0.05, seed=77)


def test_bounded_wait_gives_up_and_reports():
    wr.delta_check_device()  # nothing pending
    wr.delta_selftest_wait(polls=1000)
    with pytest.raises(wr.DeltaError) as ei:
        wr.delta_check_device()
    assert ei.value.status == wr.DELTA_ERR_CUDA
    assert "gave up" in str(ei.value) and "role 7" in str(ei.value)
    wr.delta_check_device()  # the record was cleared
    # the context is still usable: the tensor-core kernel matches the oracle
    w = small()
    inp = synth.fwd_inputs(w)
    out, hT = gpu_fwd(inp, w)
    check_full(inp, w, out, hT)


def test_injected_failure_then_recovery():
    w = small()
    inp = synth.fwd_inputs(w)
    dev = torch.device("cuda")
    args = [None if inp[n] is None else inp[n].to(dev) for n in ("q", "k", "v", "beta", "g", "h0")]
    wr.delta_inject_failure(1)
    try:
        with pytest.raises(wr.DeltaError) as ei:
            wr.delta_fwd(*args, n_h=w.n_h, chunk=w.chunk)
        assert ei.value.status == wr.DELTA_ERR_CUDA and "injected" in str(ei.value)
    finally:
        wr.delta_inject_failure(0)
    out, hT = gpu_fwd(inp, w)
    check_full(inp, w, out, hT)
