"""weight_rnn_gb300 -- delta-rule linear attention forward for one GB300.

A thin Python binding over the C ABI of ``libdelta.so`` (declared in
``include/delta.h``).  The functions keep the ABI's names and only marshal
arguments: shape/dtype checks, output allocation through PyTorch, the
current CUDA stream, and status-to-exception mapping.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback, and a
missing library raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["delta_fwd", "delta_bwd", "delta_fwd_kda", "delta_step_kda", "delta_prologue",
           "delta_fwd_prologue", "delta_step_prologue",
           "delta_fwd_static_scratch", "delta_state_erank",
           "delta_attention_map", "delta_ut_transform", "delta_fwd_with_ut", "delta_step",
           "fwd_launches", "delta_status_string", "delta_last_error",
           "delta_check_device", "delta_inject_failure", "delta_selftest_wait",
           "delta_version", "DeltaError", "library_path", "load_library",
           "DELTA_OK", "DELTA_ERR_INVALID", "DELTA_ERR_UNSUPPORTED",
           "DELTA_ERR_ALIGN", "DELTA_ERR_CUDA", "DELTA_F32", "DELTA_BF16",
           "DELTA_BETA_SIGMOID", "DELTA_BETA_2SIGMOID", "EXPORTED_SYMBOLS"]

DELTA_OK = 0
DELTA_ERR_INVALID = -1
DELTA_ERR_UNSUPPORTED = -2
DELTA_ERR_ALIGN = -3
DELTA_ERR_CUDA = -4
DELTA_F32 = 0
DELTA_BF16 = 1
DELTA_BETA_SIGMOID = 0
DELTA_BETA_2SIGMOID = 1
_BETA_MAPS = {"sigmoid": DELTA_BETA_SIGMOID, "2sigmoid": DELTA_BETA_2SIGMOID}

#: every extern "C" entry point include/delta.h declares
EXPORTED_SYMBOLS = ("delta_fwd", "delta_bwd", "delta_fwd_kda", "delta_step_kda", "delta_prologue",
                    "delta_fwd_prologue", "delta_fwd_static_scratch",
                    "delta_ut_transform", "delta_fwd_with_ut",
                    "delta_fwd_kernel_count", "delta_step", "delta_step_prologue",
                    "delta_status_string",
                    "delta_last_error", "delta_check_device", "delta_version",
                    "delta_inject_failure", "delta_selftest_wait", "delta_state_erank",
                    "delta_attention_map")

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class DeltaError(RuntimeError):
    """A libdelta call returned a non-OK status."""

    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{delta_status_string(status)} ({status}): {detail}")


def library_path() -> str:
    return os.path.join(_HERE, "libdelta.so")


def load_library():
    """Open libdelta.so and declare the ABI; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m weight_rnn_gb300.build` "
                "(the CUDA library is required; there is no fallback)")
        lib = ctypes.CDLL(path)
        p, i = ctypes.c_void_p, ctypes.c_int
        lib.delta_fwd.restype = i
        lib.delta_fwd.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, i, i, i, p]
        lib.delta_bwd.restype = i
        lib.delta_bwd.argtypes = [p] * 14 + [i] * 7 + [p]
        lib.delta_fwd_kda.restype = i
        lib.delta_fwd_kda.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, i, i, i, p]
        lib.delta_step_kda.restype = i
        lib.delta_step_kda.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, p]
        lib.delta_prologue.restype = i
        lib.delta_prologue.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, p]
        lib.delta_fwd_prologue.restype = i
        lib.delta_fwd_prologue.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, i, i, i, i, p]
        lib.delta_fwd_static_scratch.restype = i
        lib.delta_fwd_static_scratch.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, i, i, i, p]
        lib.delta_state_erank.restype = i
        lib.delta_state_erank.argtypes = [p, p, i, i, i, i, p]
        lib.delta_attention_map.restype = i
        lib.delta_attention_map.argtypes = [p, p, p, p, p, i, i, i, i, i, p]
        lib.delta_ut_transform.restype = i
        lib.delta_ut_transform.argtypes = [p, p, p, p, i, i, i, i, i, i, i, p]
        lib.delta_fwd_with_ut.restype = i
        lib.delta_fwd_with_ut.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, i, i, i, p]
        lib.delta_fwd_kernel_count.restype = i
        lib.delta_fwd_kernel_count.argtypes = [i, i, i, i, i, i, i, i]
        lib.delta_step.restype = i
        lib.delta_step.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, p]
        lib.delta_step_prologue.restype = i
        lib.delta_step_prologue.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, i, p]
        lib.delta_status_string.restype = ctypes.c_char_p
        lib.delta_status_string.argtypes = [i]
        lib.delta_last_error.restype = ctypes.c_char_p
        lib.delta_last_error.argtypes = []
        lib.delta_version.restype = i
        lib.delta_version.argtypes = []
        lib.delta_check_device.restype = i
        lib.delta_check_device.argtypes = []
        lib.delta_inject_failure.restype = i
        lib.delta_inject_failure.argtypes = [i]
        lib.delta_selftest_wait.restype = i
        lib.delta_selftest_wait.argtypes = [i, ctypes.c_void_p]
        _lib = lib
        return lib


def delta_status_string(status: int) -> str:
    return load_library().delta_status_string(int(status)).decode()


def delta_last_error() -> str:
    return load_library().delta_last_error().decode()


def delta_version() -> int:
    return int(load_library().delta_version())


def delta_check_device() -> None:
    """Synchronise the device and raise DeltaError if a library kernel gave up
    on one of its bounded internal waits since the last check."""
    st = load_library().delta_check_device()
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())


def delta_inject_failure(count: int) -> None:
    """Test hook: the next ``count`` delta_fwd / delta_step calls fail with
    DELTA_ERR_CUDA after validating their arguments, before any launch."""
    st = load_library().delta_inject_failure(int(count))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())


def delta_selftest_wait(polls: int = 1000, stream=None, device=None) -> None:
    """Enqueue one warp that gives up on a barrier nothing completes (after
    ``polls`` tries) and records that in the device error word, which the
    next delta_check_device() reports."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    st = load_library().delta_selftest_wait(int(polls), _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return DELTA_BF16
    if dt == torch.float32:
        return DELTA_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {dt}")


def _check(t, name, shape, dtype, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def delta_fwd(q, k, v, beta, g=None, h0=None, out=None, hT=None, *, n_h=1,
              chunk=64, want_state=True, stream=None):
    """Chunked forward of Gated DeltaProduct (DeltaNet for n_h = 1, g = None).

    q [B,T,H,dk]; k [B,T,n_h,H,dk] (or [B,T,H,dk] when n_h = 1);
    v [B,T,n_h,H,dv] (or [B,T,H,dv]); beta [B,T,n_h,H] (or [B,T,H]) float32;
    g [B,T,H] float32 linear gate or None; h0 [B,H,dk,dv] float32 or None.
    q/k/v share one dtype (bfloat16 or float32), which ``out`` takes too.
    Returns ``(out [B,T,H,dv], hT [B,H,dk,dv] float32 or None)``; ``hT`` may be
    passed as ``h0`` to update the state in place.
    """
    lib = load_library()
    B, T, H, dk = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("delta_fwd needs CUDA tensors")
    dt = q.dtype
    code = _dtype_code(dt)
    if n_h == 1 and k.dim() == 4:
        kshape, vshape, bshape = (B, T, H, dk), (B, T, H, v.shape[-1]), (B, T, H)
    else:
        kshape, vshape, bshape = (B, T, n_h, H, dk), (B, T, n_h, H, v.shape[-1]), (B, T, n_h, H)
    dv = v.shape[-1]
    _check(q, "q", (B, T, H, dk), dt, dev)
    _check(k, "k", kshape, dt, dev)
    _check(v, "v", vshape, dt, dev)
    _check(beta, "beta", bshape, torch.float32, dev)
    _check(g, "g", (B, T, H), torch.float32, dev)
    _check(h0, "h0", (B, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=dt, device=dev)
    _check(out, "out", (B, T, H, dv), dt, dev)
    if hT is None and want_state:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    _check(hT, "hT", (B, H, dk, dv), torch.float32, dev)
    st = lib.delta_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                       _ptr(out), _ptr(hT), B, H, T, dk, dv, n_h, chunk, code,
                       _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return out, hT


def delta_bwd(q, k, v, beta, g, h0, dout, dhT=None, *, n_h=1, want_dh0=True, stream=None):
    """Gradients of ``delta_fwd``'s out and hT (``delta_bwd``): given dout
    [B,T,H,dv] (q's dtype) and dhT [B,H,dk,dv] float32 or None, returns
    ``(dq, dk, dv, dbeta, dg, dh0)`` in float32 with the shapes of q, k, v,
    beta, g (None without g) and h0 (None unless ``want_dh0``)."""
    lib = load_library()
    B, T, H, dk = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("delta_bwd needs CUDA tensors")
    dt = q.dtype
    code = _dtype_code(dt)
    if n_h == 1 and k.dim() == 4:
        kshape, vshape, bshape = (B, T, H, dk), (B, T, H, v.shape[-1]), (B, T, H)
    else:
        kshape, vshape, bshape = (B, T, n_h, H, dk), (B, T, n_h, H, v.shape[-1]), (B, T, n_h, H)
    dv = v.shape[-1]
    _check(q, "q", (B, T, H, dk), dt, dev)
    _check(k, "k", kshape, dt, dev)
    _check(v, "v", vshape, dt, dev)
    _check(beta, "beta", bshape, torch.float32, dev)
    _check(g, "g", (B, T, H), torch.float32, dev)
    _check(h0, "h0", (B, H, dk, dv), torch.float32, dev)
    _check(dout, "dout", (B, T, H, dv), dt, dev)
    _check(dhT, "dhT", (B, H, dk, dv), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    gq, gk, gv = torch.empty((B, T, H, dk), **f32), torch.empty(kshape, **f32), torch.empty(vshape, **f32)
    gb = torch.empty(bshape, **f32)
    gg = None if g is None else torch.empty((B, T, H), **f32)
    gh0 = torch.empty((B, H, dk, dv), **f32) if want_dh0 else None
    st = lib.delta_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0), _ptr(dout), _ptr(dhT),
                       _ptr(gq), _ptr(gk), _ptr(gv), _ptr(gb), _ptr(gg), _ptr(gh0),
                       B, H, T, dk, dv, n_h, code, _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return gq, gk, gv, gb, gg, gh0


def delta_fwd_kda(q, k, v, beta, alpha, h0=None, out=None, hT=None, *, n_h=1, chunk=64,
                  want_state=True, stream=None):
    """Chunked forward with a channel-wise gate (``delta_fwd_kda``): alpha
    [B,T,H,dk] float32 decays each key row of the state, in place of g.
    Other shapes and results as in ``delta_fwd``."""
    lib = load_library()
    B, T, H, dk = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("delta_fwd_kda needs CUDA tensors")
    dt = q.dtype
    code = _dtype_code(dt)
    if n_h == 1 and k.dim() == 4:
        kshape, vshape, bshape = (B, T, H, dk), (B, T, H, v.shape[-1]), (B, T, H)
    else:
        kshape, vshape, bshape = (B, T, n_h, H, dk), (B, T, n_h, H, v.shape[-1]), (B, T, n_h, H)
    dv = v.shape[-1]
    _check(q, "q", (B, T, H, dk), dt, dev)
    _check(k, "k", kshape, dt, dev)
    _check(v, "v", vshape, dt, dev)
    _check(beta, "beta", bshape, torch.float32, dev)
    _check(alpha, "alpha", (B, T, H, dk), torch.float32, dev)
    _check(h0, "h0", (B, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=dt, device=dev)
    _check(out, "out", (B, T, H, dv), dt, dev)
    if hT is None and want_state:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    _check(hT, "hT", (B, H, dk, dv), torch.float32, dev)
    st = lib.delta_fwd_kda(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(alpha), _ptr(h0),
                           _ptr(out), _ptr(hT), B, H, T, dk, dv, n_h, chunk, code,
                           _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return out, hT


def delta_step_kda(q, k, v, beta, alpha, state, out=None, *, n_h=1, stream=None):
    """One decode token with a channel-wise gate (``delta_step_kda``): alpha
    [B,H,dk] float32 in place of g; ``state`` is updated in place."""
    lib = load_library()
    B, H, dk = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("delta_step_kda needs CUDA tensors")
    dt = q.dtype
    code = _dtype_code(dt)
    dv = v.shape[-1]
    _check(q, "q", (B, H, dk), dt, dev)
    _check(k, "k", (B, n_h, H, dk), dt, dev)
    _check(v, "v", (B, n_h, H, dv), dt, dev)
    _check(beta, "beta", (B, n_h, H), torch.float32, dev)
    _check(alpha, "alpha", (B, H, dk), torch.float32, dev)
    _check(state, "state", (B, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((B, H, dv), dtype=dt, device=dev)
    _check(out, "out", (B, H, dv), dt, dev)
    st = lib.delta_step_kda(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(alpha), _ptr(state),
                            _ptr(out), B, H, dk, dv, n_h, code, _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return out


def _beta_map(beta_map):
    if beta_map not in _BETA_MAPS:
        raise ValueError(f"beta_map {beta_map!r} is not 'sigmoid' or '2sigmoid'")
    return _BETA_MAPS[beta_map]


def delta_prologue(q_raw, k_raw, beta_raw, *, n_h=1, beta_map="sigmoid", stream=None):
    """The input prologue on its own (``delta_prologue``): returns
    ``(q, k, beta)`` with q and k through SiLU and an L2 norm over the key
    dimension (in the input dtype) and beta through ``beta_map`` (float32).
    q_raw [B,T,H,dk]; k_raw [B,T,n_h,H,dk] (or [B,T,H,dk] when n_h = 1);
    beta_raw [B,T,n_h,H] (or [B,T,H]) float32."""
    lib = load_library()
    code_map = _beta_map(beta_map)
    B, T, H, dk = q_raw.shape
    dev = q_raw.device
    if dev.type != "cuda":
        raise ValueError("delta_prologue needs CUDA tensors")
    dt = q_raw.dtype
    code = _dtype_code(dt)
    if n_h == 1 and k_raw.dim() == 4:
        kshape, bshape = (B, T, H, dk), (B, T, H)
    else:
        kshape, bshape = (B, T, n_h, H, dk), (B, T, n_h, H)
    _check(q_raw, "q_raw", (B, T, H, dk), dt, dev)
    _check(k_raw, "k_raw", kshape, dt, dev)
    _check(beta_raw, "beta_raw", bshape, torch.float32, dev)
    q = torch.empty_like(q_raw)
    k = torch.empty_like(k_raw)
    beta = torch.empty_like(beta_raw)
    st = lib.delta_prologue(_ptr(q_raw), _ptr(k_raw), _ptr(beta_raw), _ptr(q), _ptr(k), _ptr(beta),
                            B, H, T, dk, n_h, code, code_map, _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return q, k, beta


def delta_fwd_prologue(q_raw, k_raw, v, beta_raw, g=None, h0=None, out=None, hT=None, *,
                       n_h=1, chunk=64, beta_map="sigmoid", want_state=True, stream=None):
    """``delta_fwd`` on raw projections (``delta_fwd_prologue``): q and k go
    through SiLU and an L2 norm over the key dimension, beta through
    ``beta_map`` ('sigmoid' or '2sigmoid'), then the forward.  Shapes and
    results as in ``delta_fwd``."""
    lib = load_library()
    code_map = _beta_map(beta_map)
    B, T, H, dk = q_raw.shape
    dev = q_raw.device
    if dev.type != "cuda":
        raise ValueError("delta_fwd_prologue needs CUDA tensors")
    dt = q_raw.dtype
    code = _dtype_code(dt)
    if n_h == 1 and k_raw.dim() == 4:
        kshape, vshape, bshape = (B, T, H, dk), (B, T, H, v.shape[-1]), (B, T, H)
    else:
        kshape, vshape, bshape = (B, T, n_h, H, dk), (B, T, n_h, H, v.shape[-1]), (B, T, n_h, H)
    dv = v.shape[-1]
    _check(q_raw, "q_raw", (B, T, H, dk), dt, dev)
    _check(k_raw, "k_raw", kshape, dt, dev)
    _check(v, "v", vshape, dt, dev)
    _check(beta_raw, "beta_raw", bshape, torch.float32, dev)
    _check(g, "g", (B, T, H), torch.float32, dev)
    _check(h0, "h0", (B, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=dt, device=dev)
    _check(out, "out", (B, T, H, dv), dt, dev)
    if hT is None and want_state:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    _check(hT, "hT", (B, H, dk, dv), torch.float32, dev)
    st = lib.delta_fwd_prologue(_ptr(q_raw), _ptr(k_raw), _ptr(v), _ptr(beta_raw), _ptr(g),
                                _ptr(h0), _ptr(out), _ptr(hT), B, H, T, dk, dv, n_h, chunk,
                                code, code_map, _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return out, hT


def delta_fwd_static_scratch(q, k, v, beta, g=None, h0=None, out=None, hT=None, *, n_h=1,
                             chunk=64, want_state=True, stream=None):
    """``delta_fwd`` that allocates no device memory: its scratch is a static
    array of the library (at most B*H*ceil(n_h*T/64) = 4096 chunks; bf16 with
    dk = dv = 128 and chunk = 64 only).  Calls that overlap in time on one
    device race on that array.  Arguments and results as in ``delta_fwd``."""
    lib = load_library()
    B, T, H, dk = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("delta_fwd_static_scratch needs CUDA tensors")
    dt = q.dtype
    code = _dtype_code(dt)
    dv = v.shape[-1]
    kshape, vshape, bshape = _kvb_shapes(k, v, beta, B, T, H, dk, n_h)
    _check(q, "q", (B, T, H, dk), dt, dev)
    _check(k, "k", kshape, dt, dev)
    _check(v, "v", vshape, dt, dev)
    _check(beta, "beta", bshape, torch.float32, dev)
    _check(g, "g", (B, T, H), torch.float32, dev)
    _check(h0, "h0", (B, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=dt, device=dev)
    _check(out, "out", (B, T, H, dv), dt, dev)
    if hT is None and want_state:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    _check(hT, "hT", (B, H, dk, dv), torch.float32, dev)
    st = lib.delta_fwd_static_scratch(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                      _ptr(h0), _ptr(out), _ptr(hT), B, H, T, dk, dv, n_h,
                                      chunk, code, _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return out, hT


def delta_state_erank(state, erank=None, *, stream=None):
    """Effective rank of each state matrix ("DeltaProduct" §4.6): state
    [B,H,dk,dv] float32 on the GPU -> erank [B,H] float32 (0 for a zero
    matrix)."""
    lib = load_library()
    B, H, dk, dv = state.shape
    dev = state.device
    if dev.type != "cuda":
        raise ValueError("delta_state_erank needs CUDA tensors")
    _check(state, "state", (B, H, dk, dv), torch.float32, dev)
    if erank is None:
        erank = torch.empty((B, H), dtype=torch.float32, device=dev)
    _check(erank, "erank", (B, H), torch.float32, dev)
    st = lib.delta_state_erank(_ptr(state), _ptr(erank), B, H, dk, dv, _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return erank


def delta_attention_map(q, k, beta, g=None, attn=None, *, stream=None):
    """The fully parallel form ([DR] §2.4, gated as in §3) for N <= 64 steps:
    q, k [B,N,H,dk] (bf16 or float32), beta [B,N,H], g [B,N,H] or None ->
    attn [B,H,N,N] float32 with o_i = sum_j attn[i, j] v_j for a zero initial
    state."""
    lib = load_library()
    B, N, H, dk = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("delta_attention_map needs CUDA tensors")
    dt = q.dtype
    _check(q, "q", (B, N, H, dk), dt, dev)
    _check(k, "k", (B, N, H, dk), dt, dev)
    _check(beta, "beta", (B, N, H), torch.float32, dev)
    _check(g, "g", (B, N, H), torch.float32, dev)
    if attn is None:
        attn = torch.empty((B, H, N, N), dtype=torch.float32, device=dev)
    _check(attn, "attn", (B, H, N, N), torch.float32, dev)
    st = lib.delta_attention_map(_ptr(q), _ptr(k), _ptr(beta), _ptr(g), _ptr(attn), B, H, N,
                                 dk, _dtype_code(dt), _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return attn


def _kvb_shapes(k, v, beta, B, T, H, dk, n_h):
    if n_h == 1 and k.dim() == 4:
        return (B, T, H, dk), (B, T, H, v.shape[-1] if v is not None else dk), (B, T, H)
    return ((B, T, n_h, H, dk), (B, T, n_h, H, v.shape[-1] if v is not None else dk),
            (B, T, n_h, H))


def delta_ut_transform(k, beta, g=None, t_mat=None, *, n_h=1, chunk=64, stream=None):
    """The intra-chunk UT transform of every chunk (``delta_ut_transform``):
    T = (I + A)^{-1} diag(beta) per 64-step chunk of the extended sequence.

    k [B,T,n_h,H,128] (or [B,T,H,128]) bfloat16; beta [B,T,n_h,H] (or
    [B,T,H]) float32; g [B,T,H] float32 or None.  Returns ``t_mat``
    [B,H,NT,64,64] bfloat16, NT = ceil(n_h * T / 64).
    """
    lib = load_library()
    B, T = k.shape[0], k.shape[1]
    H, dk = k.shape[-2], k.shape[-1]
    dev = k.device
    if dev.type != "cuda":
        raise ValueError("delta_ut_transform needs CUDA tensors")
    code = _dtype_code(k.dtype)
    kshape, _, bshape = _kvb_shapes(k, None, beta, B, T, H, dk, n_h)
    _check(k, "k", kshape, k.dtype, dev)
    _check(beta, "beta", bshape, torch.float32, dev)
    _check(g, "g", (B, T, H), torch.float32, dev)
    nt = -(-(n_h * T) // chunk)
    if t_mat is None:
        t_mat = torch.empty((B, H, nt, chunk, chunk), dtype=torch.bfloat16, device=dev)
    _check(t_mat, "t_mat", (B, H, nt, chunk, chunk), torch.bfloat16, dev)
    st = lib.delta_ut_transform(_ptr(k), _ptr(beta), _ptr(g), _ptr(t_mat), B, H, T, dk, n_h,
                                chunk, code, _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return t_mat


def delta_fwd_with_ut(q, k, v, beta, g, h0, t_mat, out=None, hT=None, *, n_h=1, chunk=64,
                      want_state=True, stream=None):
    """The state pass alone (``delta_fwd_with_ut``), given the ``t_mat`` that
    ``delta_ut_transform`` returned for the same k, beta and g.  Arguments and
    results as in ``delta_fwd``."""
    lib = load_library()
    B, T, H, dk = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("delta_fwd_with_ut needs CUDA tensors")
    dt = q.dtype
    code = _dtype_code(dt)
    dv = v.shape[-1]
    kshape, vshape, bshape = _kvb_shapes(k, v, beta, B, T, H, dk, n_h)
    _check(q, "q", (B, T, H, dk), dt, dev)
    _check(k, "k", kshape, dt, dev)
    _check(v, "v", vshape, dt, dev)
    _check(beta, "beta", bshape, torch.float32, dev)
    _check(g, "g", (B, T, H), torch.float32, dev)
    _check(h0, "h0", (B, H, dk, dv), torch.float32, dev)
    nt = -(-(n_h * T) // chunk)
    _check(t_mat, "t_mat", (B, H, nt, chunk, chunk), torch.bfloat16, dev)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=dt, device=dev)
    _check(out, "out", (B, T, H, dv), dt, dev)
    if hT is None and want_state:
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    _check(hT, "hT", (B, H, dk, dv), torch.float32, dev)
    st = lib.delta_fwd_with_ut(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
                               _ptr(t_mat), _ptr(out), _ptr(hT), B, H, T, dk, dv, n_h, chunk,
                               code, _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return out, hT


def fwd_launches(B, H, T, dk, dv, n_h, chunk, dtype) -> int:
    """Kernels one ``delta_fwd`` call with these sizes enqueues
    (``delta_fwd_kernel_count``); raises if the sizes are rejected."""
    n = load_library().delta_fwd_kernel_count(B, H, T, dk, dv, n_h, chunk, _dtype_code(dtype))
    if n < 0:
        raise DeltaError(DELTA_ERR_UNSUPPORTED, "sizes rejected by delta_fwd")
    return n


def delta_step(q, k, v, beta, g, state, out=None, *, n_h=1, stream=None):
    """One decode token; ``state`` [B,H,dk,dv] float32 is updated in place.

    q [B,H,dk]; k [B,n_h,H,dk]; v [B,n_h,H,dv]; beta [B,n_h,H] float32;
    g [B,H] float32 or None.  Returns ``out`` [B,H,dv] in q's dtype.
    """
    lib = load_library()
    B, H, dk = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("delta_step needs CUDA tensors")
    dt = q.dtype
    code = _dtype_code(dt)
    dv = v.shape[-1]
    _check(q, "q", (B, H, dk), dt, dev)
    _check(k, "k", (B, n_h, H, dk), dt, dev)
    _check(v, "v", (B, n_h, H, dv), dt, dev)
    _check(beta, "beta", (B, n_h, H), torch.float32, dev)
    _check(g, "g", (B, H), torch.float32, dev)
    _check(state, "state", (B, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((B, H, dv), dtype=dt, device=dev)
    _check(out, "out", (B, H, dv), dt, dev)
    st = lib.delta_step(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(state),
                        _ptr(out), B, H, dk, dv, n_h, code, _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return out


def delta_step_prologue(q_raw, k_raw, v, beta_raw, g, state, out=None, *, n_h=1,
                        beta_map="sigmoid", stream=None):
    """``delta_step`` on raw projections (``delta_step_prologue``): the input
    prologue of ``delta_fwd_prologue`` runs inside the decode kernel.  Shapes
    and results as in ``delta_step``."""
    lib = load_library()
    code_map = _beta_map(beta_map)
    B, H, dk = q_raw.shape
    dev = q_raw.device
    if dev.type != "cuda":
        raise ValueError("delta_step_prologue needs CUDA tensors")
    dt = q_raw.dtype
    code = _dtype_code(dt)
    dv = v.shape[-1]
    _check(q_raw, "q_raw", (B, H, dk), dt, dev)
    _check(k_raw, "k_raw", (B, n_h, H, dk), dt, dev)
    _check(v, "v", (B, n_h, H, dv), dt, dev)
    _check(beta_raw, "beta_raw", (B, n_h, H), torch.float32, dev)
    _check(g, "g", (B, H), torch.float32, dev)
    _check(state, "state", (B, H, dk, dv), torch.float32, dev)
    if out is None:
        out = torch.empty((B, H, dv), dtype=dt, device=dev)
    _check(out, "out", (B, H, dv), dt, dev)
    st = lib.delta_step_prologue(_ptr(q_raw), _ptr(k_raw), _ptr(v), _ptr(beta_raw), _ptr(g),
                                 _ptr(state), _ptr(out), B, H, dk, dv, n_h, code, code_map,
                                 _stream(dev, stream))
    if st != DELTA_OK:
        raise DeltaError(st, delta_last_error())
    return out
