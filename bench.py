#!/usr/bin/env python
"""Throughput of the delta-rule forward on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 2|3|4|5]

A step is one pass of the hot path over one batch of synthetic input: one
``delta_fwd`` call on the DeltaNet workload B8 H16 T4096 dk=dv=128 bf16,
chunk 64 (the default; ``--workload`` 3/4 select the gated and DeltaProduct
workloads, 5 the B256 x H32 decode step).  Inputs are resident in HBM and
larger than L2 (403 MB of q/k/v per step for the default workload), so no
flush is needed between steps.

Reported besides tokens/s: the roofline of the kernel (achieved GB/s over
algorithmic bytes vs the measured HBM peak), the end-to-end rate through the
public API with host buffers (copies inside the timed region), the CPU
oracle's rate on a bounded sample of the same workload, SM clocks sampled
during the timed region, and the number of kernels launched.

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
GPU with its own seed (weak scaling over independent heads, no collective on
the data path); timing is barrier-bracketed and the max over ranks is taken.
``--impl reference`` times the float64 CPU oracle on the host cores instead
(rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from weight_rnn_gb300 import synth  # noqa: E402

METRIC = "delta fwd tokens/s (B·H·T/s) at dk=dv=128; % of tensor/HBM roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "fwd": ["weight_rnn_gb300/csrc/chunk_tc.cu", "weight_rnn_gb300/csrc/chunk_generic.cu"],
    "step": ["weight_rnn_gb300/csrc/step.cu"],
}


# --------------------------------------------------------------------------- utils
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(kind):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def algorithmic_bytes(w: synth.Workload) -> int:
    """HBM bytes one forward must move: q, k, v, beta, g, out, h0, hT."""
    e = 2 if w.dtype == "bf16" else 4
    BT = w.B * w.T * w.H
    n = BT * w.dk * e + BT * w.n_h * (w.dk + w.dv) * e + BT * w.n_h * 4 + BT * w.dv * e
    if w.gated:
        n += BT * 4
    state = w.B * w.H * w.dk * w.dv * 4
    n += state  # hT
    if w.h0_std > 0:
        n += state
    return n


def algorithmic_flops(w: synth.Workload) -> float:
    """Dense-contraction flops of the chunked algorithm (triangles counted
    half, readout only for real output rows), per forward."""
    C, dk, dv, n_h = w.chunk, w.dk, w.dv, w.n_h
    L = w.T * n_h
    chunks = -(-L // C)
    rows_out = C / n_h
    mac = (C * (C - 1) / 2 * dk          # strictly lower K K^T
           + C ** 3 / 6                   # triangular solve
           + C * (C + 1) / 2 * (dk + dv)  # W = T K, U = T V
           + C * dk * dv                  # W S
           + rows_out * dk * dv           # Q S (readout rows)
           + rows_out * (C + 1) / 2 * (dk + dv)  # Q K^T masked, P Vt
           + C * dk * dv)                 # K^T Vt
    return 2.0 * mac * chunks * w.B * w.H


def step_bytes(w: synth.Workload) -> int:
    e = 2 if w.dtype == "bf16" else 4
    BH = w.B * w.H
    n = BH * (w.dk + w.n_h * (w.dk + w.dv) + w.dv) * e + BH * w.n_h * 4
    if w.gated:
        n += BH * 4
    return n + 2 * BH * w.dk * w.dv * 4


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.lines = []
        self.bus = None
        try:
            pr = torch.cuda.get_device_properties(device)
            self.bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
        except Exception:
            self.bus = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.bus:
            cmd += ["-i", self.bus]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names[1:], parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- dist
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float, device=None) -> float:
        if not self.pg:
            return x
        t = torch.tensor([x], dtype=torch.float64,
                         device=device if device is not None else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# --------------------------------------------------------------------------- oracle leg
def oracle_sample_rate(w: synth.Workload, inp, heads: int, threads: int):
    """Time the float64 oracle (as it stands) on the first `heads` heads."""
    import oracle  # test infrastructure: only this leg of the bench uses it

    pairs = [(b, h) for b in range(w.B) for h in range(w.H)][:heads]
    n = len(pairs)
    f = lambda t: t.float().numpy()
    # the sampled heads become a batch of n single-head sequences
    q = np.stack([f(inp["q"][b, :, h]) for b, h in pairs]).reshape(n, w.T, 1, w.dk)
    k = np.stack([f(inp["k"][b, :, :, h]) for b, h in pairs]).reshape(n, w.T, w.n_h, 1, w.dk)
    v = np.stack([f(inp["v"][b, :, :, h]) for b, h in pairs]).reshape(n, w.T, w.n_h, 1, w.dv)
    beta = np.stack([f(inp["beta"][b, :, :, h]) for b, h in pairs]).reshape(n, w.T, w.n_h, 1)
    g = (None if inp["g"] is None else
         np.stack([f(inp["g"][b, :, h]) for b, h in pairs]).reshape(n, w.T, 1))
    h0 = (None if inp["h0"] is None else
          np.stack([f(inp["h0"][b, h]) for b, h in pairs]).reshape(n, 1, w.dk, w.dv))
    t0 = time.perf_counter()
    oracle.fwd(q, k, v, beta, g, h0, n_h=w.n_h, threads=threads, want_state=True)
    dt = time.perf_counter() - t0
    return len(pairs) * w.T / dt, dt, len(pairs)


def run_reference(args, w, dist):
    if dist.rank != 0:
        return 0
    threads = os.cpu_count() or 1
    inp = synth.fwd_inputs(w.with_(B=1, H=min(w.H, max(1, threads))), seed=w.seed)
    wsmall = w.with_(B=1, H=min(w.H, max(1, threads)))
    heads = wsmall.H
    for _ in range(args.warmup):
        oracle_sample_rate(wsmall, inp, heads, threads)
    tot_t, tot_tok = 0.0, 0
    for _ in range(args.steps):
        _, dt, n = oracle_sample_rate(wsmall, inp, heads, threads)
        tot_t += dt
        tot_tok += n * w.T
    value = tot_tok / tot_t
    sample = (f"{heads} heads x {w.T} tokens per step (of {w.B * w.H} heads) of "
              f"{w.name}, float64, {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, args):
    c = {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
         "n_h": w.n_h, "chunk": w.chunk, "gated": w.gated, "h0": w.h0_std > 0,
         "io_dtype": w.dtype, "parallelism": f"replicas x{args.gpus} over (b,h)"}
    if w.calls:
        c.update({"T": 1, "calls_per_step": 1})
        c["l2"] = "state 512 MiB > L2 (129 MB): no flush needed"
    else:
        c["l2"] = "inputs larger than L2 (129 MB) every step: no flush needed"
    return c


# --------------------------------------------------------------------------- ours
def read_traffic(kind, workload_name):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(kind)
    if not ent or ent.get("source_sha") != source_sha(kind):
        return None
    if ent.get("workload") != workload_name:
        return None
    return ent.get("dram_bytes_per_launch")


def run_ours(args, w, dist):
    import weight_rnn_gb300 as wr

    wr.load_library()
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    decode = bool(w.calls)

    # ---- inputs (per-rank seed: each GPU owns its own heads) ----
    if decode:
        host = synth.step_inputs(w, dist.rank)
        names = ("q", "k", "v", "beta", "g")
    else:
        host = synth.fwd_inputs(w, seed=w.seed + 7919 * dist.rank)
        names = ("q", "k", "v", "beta", "g", "h0")
    d = {n: (None if host[n] is None else host[n].to(dev)) for n in names}
    if decode:
        state = torch.zeros(w.B, w.H, w.dk, w.dv, device=dev)
        out = torch.empty(w.B, w.H, w.dv, dtype=synth.torch_dtype(w.dtype), device=dev)

        def step():
            wr.delta_step(d["q"], d["k"], d["v"], d["beta"], d["g"], state, out,
                          n_h=w.n_h)
        tokens = w.B * w.H
        kbytes = step_bytes(w)
        kflops = None
        kind = "step"
    else:
        out = torch.empty(w.B, w.T, w.H, w.dv, dtype=synth.torch_dtype(w.dtype), device=dev)
        hT = torch.empty(w.B, w.H, w.dk, w.dv, device=dev)

        def step():
            wr.delta_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], out, hT,
                         n_h=w.n_h, chunk=w.chunk)
        tokens = w.tokens
        kbytes = algorithmic_bytes(w)
        kflops = algorithmic_flops(w)
        kind = "fwd"

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # ---- device-resident timed region ----
    clocks = ClockSampler(dev) if dist.local == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    clock_rec = clocks.stop() if clocks else None
    elapsed = t_start.elapsed_time(t_end) / 1e3
    kernel_s = sum(a.elapsed_time(b) for a, b in ev) / 1e3 / args.steps
    elapsed = dist.max(elapsed, dev)
    kernel_s = dist.max(kernel_s, dev)
    ms_per_step = 1e3 * elapsed / args.steps
    value = tokens * dist.world * args.steps / elapsed

    # ---- end to end through the public API with pinned host buffers ----
    pinned = {n: (None if host[n] is None else host[n].pin_memory()) for n in names}
    h2d = sum(t.numel() * t.element_size() for t in pinned.values() if t is not None)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    if decode:
        state_h = torch.empty(state.shape, dtype=state.dtype).pin_memory()
        d2h = out_h.numel() * out_h.element_size()
    else:
        hT_h = torch.empty(hT.shape, dtype=hT.dtype).pin_memory()
        d2h = (out_h.numel() * out_h.element_size() + hT_h.numel() * hT_h.element_size())

    def e2e_step():
        for n in names:
            if pinned[n] is not None:
                d[n].copy_(pinned[n], non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)
        if not decode:
            hT_h.copy_(hT, non_blocking=True)

    for _ in range(min(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_s = dist.max(e0.elapsed_time(e1) / 1e3, dev)
    e2e_value = tokens * dist.world * args.steps / e2e_s

    # ---- roofline of the (only) kernel of a step ----
    hbm = float(peaks["hbm_gbs"])
    achieved = kbytes / kernel_s / 1e9
    t_hbm = kbytes / (hbm * 1e9)
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": read_traffic(kind, w.name),
            "algorithmic_bytes_per_launch": kbytes,
            "kernel_us": kernel_s * 1e6, "peak_source": f"hbm_gbs of {peak_src}"}
    if kflops is not None:
        tc = float(peaks["bf16_tflops"])
        t_tc = kflops / (tc * 1e12)
        roof["tensor_tflops_achieved"] = kflops / kernel_s / 1e12
        roof["tensor_frac"] = (kflops / kernel_s / 1e12) / tc
        roof["roofline_time_us"] = max(t_hbm, t_tc) * 1e6
        roof["roofline_frac"] = max(t_hbm, t_tc) / kernel_s
        if t_tc > t_hbm:
            roof.update({"bound": "tensor", "achieved": kflops / kernel_s / 1e12,
                         "peak": tc, "unit": "TFLOP/s", "frac": roof["tensor_frac"],
                         "peak_source": f"bf16_tflops of {peak_src}"})

    # ---- CPU oracle on a bounded sample (rank 0, N = 1 only) ----
    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline and not decode:
        threads = os.cpu_count() or 1
        # every head of the workload: ~13 s of CPU work at B8 H16 T4096
        heads = w.B * w.H
        rate, dt, n = oracle_sample_rate(w, host, heads, threads)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{n} of {w.B * w.H} heads x {w.T} tokens of {w.name} "
                         f"({dt:.1f} s wall, float64)"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config_of(w, args), "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": clock_rec, "gpu_launches": args.steps,
        "gpu": torch.cuda.get_device_name(dev),
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2, choices=[2, 3, 4, 5])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    # at least 3 untimed warm-up steps, whatever is asked
    args.warmup = max(args.warmup, 3)
    w = synth.WORKLOADS[args.workload]
    dist = Dist()
    if args.impl == "reference":
        return run_reference(args, w, dist)
    return run_ours(args, w, dist)


if __name__ == "__main__":
    sys.exit(main())
