"""Seeded synthetic inputs for delta-rule attention workloads.

This module only draws random numbers with the shapes and value
distributions of the workloads; it holds none of the method's arithmetic.
Both the test suite (GPU path and CPU oracle alike) and ``bench.py`` draw
their inputs here.

Recipe: a ``torch.Generator`` on the CPU seeded per workload, float32 draws in
the fixed order q, k, v, beta, g, h0, every element i.i.d., then a cast of
q/k/v to the I/O dtype.  The distributions follow the model layer the pages
describe: keys and queries are SiLU'd and L2-normalised per token and head
("08 · linear 路线（三）：delta rule 与 DPLR 统一框架", §3 layer design;
"DeltaProduct …" reading notes §2.2), beta = sigmoid (or 2*sigmoid to allow
negative eigenvalues, "DeltaProduct …" §2.2), and the gate is a Mamba-2 style
exp(-softplus(x) * 0.1) per token and head.

The SiLU and normalisation here only give the forward's inputs the shape of
that layer's outputs (the forward takes normalised keys).  The input
prologue, which computes the same maps as part of the method, is implemented
separately by its kernel and by the oracle, and both are tested on raw draws
that do not pass through this module.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    n_h: int
    chunk: int
    dtype: str            # "bf16" or "f32" for q, k, v and out
    qk: str               # "l2_normal" | "l2_silu"
    beta_scale: float     # 1 -> sigmoid, 2 -> 2*sigmoid
    gated: bool
    h0_std: float         # 0 -> no initial state
    seed: int
    calls: int = 0        # decode workloads: number of successive steps

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.T


WORKLOADS = {
    1: Workload("deltanet_smoke_b1_h1_t64_d16_f32", 1, 1, 64, 16, 16, 1, 16,
                "f32", "l2_normal", 1.0, False, 0.0, 1001),
    2: Workload("deltanet_b8_h16_t4096_d128_bf16", 8, 16, 4096, 128, 128, 1, 64,
                "bf16", "l2_silu", 1.0, False, 0.0, 1002),
    3: Workload("gated_deltanet_b4_h32_t8192_d128_bf16_h0", 4, 32, 8192, 128, 128,
                1, 64, "bf16", "l2_silu", 1.0, True, 0.02, 1003),
    4: Workload("gated_deltaproduct_b4_h16_t4096_nh3_d128_bf16", 4, 16, 4096, 128,
                128, 3, 64, "bf16", "l2_silu", 2.0, True, 0.0, 1004),
    5: Workload("decode_b256_h32_d128_nh2_f32_1024calls", 256, 32, 1, 128, 128, 2,
                0, "f32", "l2_normal", 1.0, True, 0.0, 1005, calls=1024),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _keys(gen, shape, kind):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if kind == "l2_silu":
        x = torch.nn.functional.silu(x)
    elif kind != "l2_normal":
        raise ValueError(kind)
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def _gate(gen, shape):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    return torch.exp(-torch.nn.functional.softplus(x) * 0.1)


def fwd_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """CPU tensors for one forward call in the library's layouts:
    q [B,T,H,dk], k [B,T,n_h,H,dk], v [B,T,n_h,H,dv] in the I/O dtype;
    beta [B,T,n_h,H] fp32; g [B,T,H] fp32 or None; h0 [B,H,dk,dv] fp32 or None.
    """
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    B, T, H, n_h, dk, dv = w.B, w.T, w.H, w.n_h, w.dk, w.dv
    q = _keys(gen, (B, T, H, dk), w.qk)
    k = _keys(gen, (B, T, n_h, H, dk), w.qk)
    v = torch.randn((B, T, n_h, H, dv), generator=gen, dtype=torch.float32)
    beta = torch.sigmoid(torch.randn((B, T, n_h, H), generator=gen)) * w.beta_scale
    g = _gate(gen, (B, T, H)) if w.gated else None
    h0 = (torch.randn((B, H, dk, dv), generator=gen) * w.h0_std
          if w.h0_std > 0 else None)
    dt = torch_dtype(w.dtype)
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), beta=beta.contiguous(),
                g=None if g is None else g.contiguous(),
                h0=None if h0 is None else h0.contiguous())


def step_seed(w: Workload, call: int) -> int:
    """Seed of decode call number ``call`` (fresh inputs every call)."""
    return w.seed * 100003 + call


def step_inputs(w: Workload, call: int) -> dict:
    """CPU tensors for one decode call: q [B,H,dk], k [B,n_h,H,dk],
    v [B,n_h,H,dv] in the I/O dtype; beta [B,n_h,H]; g [B,H] or None."""
    gen = torch.Generator().manual_seed(step_seed(w, call))
    B, H, n_h, dk, dv = w.B, w.H, w.n_h, w.dk, w.dv
    q = _keys(gen, (B, H, dk), w.qk)
    k = _keys(gen, (B, n_h, H, dk), w.qk)
    v = torch.randn((B, n_h, H, dv), generator=gen, dtype=torch.float32)
    beta = torch.sigmoid(torch.randn((B, n_h, H), generator=gen)) * w.beta_scale
    g = _gate(gen, (B, H)) if w.gated else None
    dt = torch_dtype(w.dtype)
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), beta=beta.contiguous(),
                g=None if g is None else g.contiguous())
