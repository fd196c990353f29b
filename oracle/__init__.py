"""CPU oracle for delta-rule linear attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (``weight_rnn_gb300``)
never imports it and fails loudly when its CUDA library is missing.

Two parts:

* ``fwd`` -- the float64 token-by-token recurrence in ``delta_oracle.c``
  (gate once per token, then ``n_h`` delta sub-steps, then the readout), loaded
  through ctypes.  Threads run over independent (b, h) heads.
* ``oracle.forms`` -- independent NumPy float64 restatements of the other
  forms the pages give (erase-write, gradient step, WY, UT/chunkwise, fully
  parallel, DPLR loop, product expansion), used to pin ``fwd`` on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "delta_oracle.c")
_LIB = os.path.join(_HERE, "libdelta_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``delta_oracle.c`` into ``libdelta_oracle.so`` next to it."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def load_library(path):
    """Open a compiled oracle library and declare its entry point."""
    lib = ctypes.CDLL(path)
    f = lib.delta_oracle_fwd
    f.restype = ctypes.c_int
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    f.argtypes = [p, p, p, p, p, p, p, p,
                  i64, i64, i64, i64, i64, i64, ctypes.c_int]
    f64 = lib.delta_oracle_fwd_state64
    f64.restype = ctypes.c_int
    f64.argtypes = list(f.argtypes)
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load_library(_LIB)
    return _lib


def _f32(x):
    if x is None:
        return None
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _shapes(q, k, v, beta, g, h0, n_h):
    B, T, H, dk = q.shape
    if k.ndim == 4:
        if n_h != 1:
            raise ValueError("k without a sub-step axis requires n_h == 1")
        k = k.reshape(B, T, 1, H, dk)
        v = v.reshape(B, T, 1, H, v.shape[-1])
        beta = beta.reshape(B, T, 1, H)
    dv = v.shape[-1]
    if k.shape != (B, T, n_h, H, dk):
        raise ValueError(f"k shape {k.shape} != {(B, T, n_h, H, dk)}")
    if v.shape != (B, T, n_h, H, dv):
        raise ValueError(f"v shape {v.shape}")
    if beta.shape != (B, T, n_h, H):
        raise ValueError(f"beta shape {beta.shape}")
    if g is not None and g.shape != (B, T, H):
        raise ValueError(f"g shape {g.shape}")
    if h0 is not None and h0.shape != (B, H, dk, dv):
        raise ValueError(f"h0 shape {h0.shape}")
    return k, v, beta, (B, T, H, dk, dv)


def fwd(q, k, v, beta, g=None, h0=None, *, n_h=1, threads=None,
        want_state=True, lib=None, state64=False):
    """Run the float64 recurrence.

    Shapes: q [B,T,H,dk]; k [B,T,n_h,H,dk]; v [B,T,n_h,H,dv];
    beta [B,T,n_h,H]; g [B,T,H] or None; h0 [B,H,dk,dv] or None.
    For ``n_h == 1`` the sub-step axis may be omitted (k [B,T,H,dk], ...).

    Token inputs are taken as float32 (every bf16/fp32 input is exact in
    float32).  h0 is taken as float32 too, unless ``state64`` is set: then it
    is read as float64, unrounded (a state carried between decode calls).
    Returns ``(out [B,T,H,dv] float64, hT [B,H,dk,dv] float64 or None)``.
    ``lib`` selects another compiled copy of the oracle (tests only).
    """
    q = _f32(q)
    k = _f32(k)
    v = _f32(v)
    beta = _f32(beta)
    g = _f32(g)
    if state64:
        h0 = None if h0 is None else np.ascontiguousarray(np.asarray(h0, dtype=np.float64))
    else:
        h0 = _f32(h0)
    k, v, beta, (B, T, H, dk, dv) = _shapes(q, k, v, beta, g, h0, n_h)
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    hT = np.zeros((B, H, dk, dv), dtype=np.float64) if want_state else None
    if threads is None:
        threads = os.cpu_count() or 1
    lib = lib or _load()
    entry = lib.delta_oracle_fwd_state64 if state64 else lib.delta_oracle_fwd
    rc = entry(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(h0),
               _ptr(out), _ptr(hT), B, H, T, dk, dv, n_h, int(threads))
    if rc != 0:
        raise RuntimeError(f"delta_oracle_fwd failed with status {rc}")
    return out, hT


def step(q, k, v, beta, g, state, *, n_h=1, threads=None, lib=None):
    """One decode step: the same recurrence with T = 1 ("08 · linear 路线（三）"
    §2.3, the recurrent form that serves decoding; the sub-steps and gate of
    "DeltaProduct" §2.6).

    q [B,H,dk]; k [B,n_h,H,dk]; v [B,n_h,H,dv]; beta [B,n_h,H]; g [B,H] or
    None; state [B,H,dk,dv] or None (=> zero).  The state is read and
    returned in float64, never rounded, so that chained calls equal one
    forward over the same tokens.  Returns ``(out [B,H,dv], new_state)``.
    """
    q = np.asarray(q)
    B, H, dk = q.shape
    dv = np.asarray(v).shape[-1]
    out, hT = fwd(q.reshape(B, 1, H, dk),
                  np.asarray(k).reshape(B, 1, n_h, H, dk),
                  np.asarray(v).reshape(B, 1, n_h, H, dv),
                  np.asarray(beta).reshape(B, 1, n_h, H),
                  None if g is None else np.asarray(g).reshape(B, 1, H),
                  state, n_h=n_h, threads=threads, lib=lib, state64=True)
    return out.reshape(B, H, dv), hT


def rel_l2(x, ref):
    """Global relative L2 error ||x - ref||_2 / ||ref||_2 over every element,
    in float64 (the reading of the pages' "rel err" taken for every parity
    tolerance).  The reference is the second argument.  If ``ref`` is all
    zero the absolute error ||x - ref||_2 is returned instead."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((x - ref).ravel())
    if den == 0.0:
        return float(num)
    return float(num / den)
