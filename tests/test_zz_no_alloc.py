"""delta_fwd_static_scratch: the tensor-core forward with its T-tile scratch in
a static device array of the library instead of an allocation.  Its results
are compared with delta_fwd's on the same inputs, within the bf16 parity
tolerance, over two calls in a row; sizes past the array are rejected before
anything is enqueued."""
import ctypes

import numpy as np
import pytest
import torch

import weight_rnn_gb300 as wr
from weight_rnn_gb300 import build as wbuild
from weight_rnn_gb300 import synth
from parity import compare, to_np

W = synth.WORKLOADS
MAX_CHUNKS = 4096  # the array: 32 MiB of 8 KiB T tiles


def _small(seed, T=200, n_h=1, gated=True, h0=0.05, B=2, H=3):
    return W[2].with_(name="static", B=B, H=H, T=T, n_h=n_h, gated=gated, h0_std=h0,
                      beta_scale=2.0 if n_h > 1 else 1.0, seed=seed)


def _on_gpu(inp):
    dev = torch.device("cuda")
    return {n: (None if inp[n] is None else inp[n].to(dev)) for n in inp}


def _both(w, d):
    """delta_fwd and the static-scratch call on the same device inputs."""
    args = (d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    ref = wr.delta_fwd(*args, n_h=w.n_h)
    got = wr.delta_fwd_static_scratch(*args, n_h=w.n_h)
    return ref, got


def _same(ref, got, what):
    compare(to_np(got[0]), to_np(ref[0]), "bf16", f"{what} out")
    compare(to_np(got[1]), to_np(ref[1]), "bf16", f"{what} hT")


@pytest.mark.gpu
@pytest.mark.parametrize("T,n_h,gated,h0", [(200, 1, True, 0.05), (130, 3, True, 0.0),
                                             (1000, 1, False, 0.0)])
def test_two_calls_in_a_row_match_delta_fwd(T, n_h, gated, h0):
    # two different problems enqueued back to back: the second call's T tiles
    # overwrite the first's in the one array, after the first call's kernels
    w1, w2 = _small(11, T, n_h, gated, h0), _small(12, T, n_h, gated, h0)
    d1, d2 = _on_gpu(synth.fwd_inputs(w1)), _on_gpu(synth.fwd_inputs(w2))
    a1 = (d1["q"], d1["k"], d1["v"], d1["beta"], d1["g"], d1["h0"])
    a2 = (d2["q"], d2["k"], d2["v"], d2["beta"], d2["g"], d2["h0"])
    got1 = wr.delta_fwd_static_scratch(*a1, n_h=n_h)
    got2 = wr.delta_fwd_static_scratch(*a2, n_h=n_h)
    ref1 = wr.delta_fwd(*a1, n_h=n_h)
    ref2 = wr.delta_fwd(*a2, n_h=n_h)
    torch.cuda.synchronize()
    wr.delta_check_device()
    _same(ref1, got1, "call 1")
    _same(ref2, got2, "call 2")


@pytest.mark.gpu
def test_largest_problem_the_array_holds():
    # B1 H32 T8192: 32 * 128 = 4096 chunks, the whole array, called twice
    w = W[3].with_(name="static_max", B=1)
    assert w.B * w.H * -(-w.T * w.n_h // 64) == MAX_CHUNKS
    d = _on_gpu(synth.fwd_inputs(w))
    ref, got = _both(w, d)
    again = wr.delta_fwd_static_scratch(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                                        n_h=w.n_h)
    torch.cuda.synchronize()
    wr.delta_check_device()
    _same(ref, got, "first")
    _same(ref, again, "second")


@pytest.mark.gpu
def test_empty_sequence_copies_the_state():
    w = _small(13, T=0)
    d = _on_gpu(synth.fwd_inputs(w.with_(T=1)))
    h0 = d["h0"]
    q, k, v, beta, g = (d[n][:, :0] for n in ("q", "k", "v", "beta", "g"))
    out, hT = wr.delta_fwd_static_scratch(q, k, v, beta, g, h0, n_h=1)
    torch.cuda.synchronize()
    assert out.numel() == 0
    assert torch.equal(hT, h0)


# --- rejections, checked before any CUDA call (no GPU needed) ---------------
def _call(lib, B, H, T, dk=128, dv=128, n_h=1, chunk=64, dtype=wr.DELTA_BF16):
    # pointers 2^40 apart: aligned, never dereferenced, never overlapping
    p = [ctypes.c_void_p((i + 1) << 40) for i in range(6)]
    return lib.delta_fwd_static_scratch(p[0], p[1], p[2], p[3], None, None, p[4], p[5],
                                        B, H, T, dk, dv, n_h, chunk, dtype, None)


def test_rejects_more_chunks_than_the_array_holds():
    wbuild.build()
    lib = wr.load_library()
    # 32 x ceil(8193 / 64) = 4128 chunks > 4096
    assert _call(lib, 1, 32, 8193) == wr.DELTA_ERR_UNSUPPORTED
    assert "4128 chunks" in wr.delta_last_error()
    # n_h counts: 1 x 16 x ceil(3 * 5462 / 64) = 4112 chunks
    assert _call(lib, 1, 16, 5462, n_h=3) == wr.DELTA_ERR_UNSUPPORTED


def test_rejects_shapes_outside_the_tensor_core_set():
    wbuild.build()
    lib = wr.load_library()
    assert _call(lib, 1, 1, 64, dk=64, dv=64) == wr.DELTA_ERR_UNSUPPORTED
    assert _call(lib, 1, 1, 64, chunk=32) == wr.DELTA_ERR_UNSUPPORTED
    assert _call(lib, 1, 1, 64, dtype=wr.DELTA_F32) == wr.DELTA_ERR_UNSUPPORTED
    assert _call(lib, -1, 1, 64) == wr.DELTA_ERR_INVALID
