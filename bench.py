#!/usr/bin/env python
"""Throughput of the delta-rule forward on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload all|2|3|4|5]

A step is one pass of the hot path over one batch of synthetic input: one
``delta_fwd`` call over a whole workload (or one ``delta_step`` call for the
decode workload).  By default every workload runs in one invocation, each
with W untimed warm-up steps and K timed steps:

  3  Gated DeltaNet      B4 H32 T8192 dk=dv=128 bf16, chunk 64, h0   (headline)
  2  DeltaNet            B8 H16 T4096 dk=dv=128 bf16, chunk 64
  4  Gated DeltaProduct  B4 H16 T4096 n_h=3 dk=dv=128 bf16, chunk 64
  5  decode step         B256 H32 dk=dv=128 n_h=2, fp32 state 512 MiB

The headline (``value``, ``roofline``, ``e2e``, ``cpu_baseline``) is the
largest dk=dv=128 forward that fits one GPU, workload 3; ``per_workload``
carries the same figures for every workload.  Inputs are resident in HBM and
larger than L2 (129 MB) every step, so no flush is needed between steps.

Reported besides tokens/s: the roofline of the step (algorithmic bytes over
the CUDA-event time of the step's kernels vs the measured HBM peak, and vs
the GB300's nominal 7.9 TB/s), the spread of the per-step kernel times, the
end-to-end rate through the public API with host buffers (copies inside the
timed region, overlapped with compute over batch slices on two streams), the
CPU oracle's rate on the headline workload (all cores and one core), SM
clocks sampled during the timed regions, and the number of kernels launched.

Under torchrun (N > 1) every rank runs the same per-GPU workloads on its own
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
import re
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
HEADLINE = 3
ORDER = (3, 2, 4, 5)
SPEC_HBM_GBS = 7900.0  # GB300 nominal HBM3e bandwidth
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "fwd": ["weight_rnn_gb300/csrc/chunk_tc.cu", "weight_rnn_gb300/csrc/ut_tc.cu"],
    "ut": ["weight_rnn_gb300/csrc/ut_tc.cu"],
    "state": ["weight_rnn_gb300/csrc/chunk_tc.cu"],
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


def _code_only(text):
    """A kernel source without its comments and blank lines, so that the hash
    below changes when the code does and not when a comment is reworded."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def source_sha(kind):
    """Hash of the code (comments aside) of the kernel sources behind `kind`;
    a traffic record counts only while its recorded hash matches."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
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


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


class NvmlPoller:
    """Read-only clock, power and clock-event-reason queries through the
    driver's NVML library (ctypes), polled about every millisecond from a
    thread, each sample tagged with whether the timed region was running.
    Any failure (no library, no device, a query error) leaves `ok` False or
    ends the polling; nothing here changes a GPU setting."""

    CLOCK_SM = 1  # nvmlClockType_t: the SM clock
    # nvmlClocksEventReasons bits that the timing rules name
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, bus_id, lib=None):
        import ctypes
        self.ct = ctypes
        self.ok = False
        self.samples = []  # (sm_mhz, max_mhz, watts, reason_bits, in_region)
        self.in_region = False
        self._stop = threading.Event()
        self.thread = None
        try:
            self.lib = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(self.h)) != 0:
                return
            self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = self.sample() is not None
        except Exception:
            self.ok = False

    def sample(self):
        ct = self.ct
        mhz, mx, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if (self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ct.byref(mhz)) != 0 or
                self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ct.byref(mx)) != 0):
            return None
        if self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw)) != 0:
            mw.value = 0
        if self._reasons(self.h, ct.byref(rs)) != 0:
            rs.value = 0
        return (float(mhz.value), float(mx.value), mw.value / 1000.0, int(rs.value))

    def _run(self):
        try:
            while not self._stop.is_set():
                smp = self.sample()
                if smp is None:
                    return
                self.samples.append(smp + (self.in_region,))
                time.sleep(0.0005)
        except Exception:
            return

    def start(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self):
        self._stop.set()
        if self.thread is not None:
            self.thread.join(timeout=5)
        try:
            self.lib.nvmlShutdown()
        except Exception:
            pass
        loaded = [x for x in self.samples if x[4]]
        use = loaded or self.samples
        reasons = sorted({name for x in use for bit, name in self.REASONS.items() if x[3] & bit})
        return {"sm_mhz": statistics.median(x[0] for x in use) if use else None,
                "sm_max_mhz": max(x[1] for x in self.samples) if self.samples else None,
                "reasons": reasons, "samples": len(self.samples),
                "samples_under_load": len(loaded), "source": "nvml, timed region"}


class ClockSampler:
    """Clock/throttle samples while the timed region runs: NVML polled about
    every millisecond (samples inside the timed region count as under load),
    else nvidia-smi at 100 ms (under load = power well above idle)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.nvml = None
        self.lines = []
        self.bus = None
        try:
            pr = torch.cuda.get_device_properties(device)
            self.bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
        except Exception:
            self.bus = None

    def region(self, running):
        """Mark the timed region (NVML samples taken inside it are under load)."""
        if self.nvml is not None:
            self.nvml.in_region = running

    def start(self):
        self.nvml = None
        if self.bus:
            try:
                nv = NvmlPoller(self.bus)
                if nv.ok:
                    nv.start()
                    self.nvml = nv
                    return
            except Exception:
                self.nvml = None
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
        if self.nvml is not None:
            try:
                return self.nvml.stop()
            except Exception:
                return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml sampling failed"],
                        "samples": 0, "samples_under_load": 0}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0, "samples_under_load": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names[1:], parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        # samples under load: power well above the first sample's, taken while
        # the GPU was still idle (before the warm-up steps)
        loaded = [s for s, p in zip(sm, power) if power and p > power[0] + 50.0]
        return {"sm_mhz": statistics.median(loaded or sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "samples_under_load": len(loaded), "source": "nvidia-smi"}


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


def cpu_baseline(w, host):
    """The oracle on the host cores: every head with all cores, and two heads
    on one core (extrapolated to the whole workload by head count)."""
    threads = os.cpu_count() or 1
    rate, dt, n = oracle_sample_rate(w, host, w.B * w.H, threads)
    rate1, dt1, n1 = oracle_sample_rate(w, host, 2, 1)
    return {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{n} of {w.B * w.H} heads x {w.T} tokens of {w.name} "
                      f"({dt:.1f} s wall, float64, {threads} threads)",
            "single_core": {"value": rate1, "unit": UNIT, "cores": 1,
                            "sample": f"{n1} heads x {w.T} tokens ({dt1:.2f} s)",
                            "whole_workload_s": w.tokens / rate1}}


def run_reference(args, dist):
    if dist.rank != 0:
        return 0
    w = synth.WORKLOADS[HEADLINE if args.workload == "all" else int(args.workload)]
    threads = os.cpu_count() or 1
    wsmall = w.with_(B=1, H=min(w.H, max(1, threads)))
    inp = synth.fwd_inputs(wsmall, seed=w.seed)
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
                         "cpu_model": cpu_model(), "sample": sample},
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
    for ent in rec.get("records", []):
        if (ent.get("kind") == kind and ent.get("workload") == workload_name
                and ent.get("source_sha") == source_sha(kind)):
            return ent.get("dram_bytes_per_launch")
    return None


def _spread(xs):
    xs = sorted(xs)
    return {"min": xs[0], "median": statistics.median(xs), "max": xs[-1]}


def measure(w, wr, dist, dev, args, peaks, peak_src, clocks_on):
    """Time one workload; returns its record (rank-max times)."""
    stream = torch.cuda.current_stream(dev)
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

        def step(dd=d, o=out, st=state, s=None):
            wr.delta_step(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], st, o,
                          n_h=w.n_h, stream=s)
        tokens = w.B * w.H
        kbytes = step_bytes(w)
        kflops = None
        kind = "step"
        launches = 1
    else:
        out = torch.empty(w.B, w.T, w.H, w.dv, dtype=synth.torch_dtype(w.dtype), device=dev)
        hT = torch.empty(w.B, w.H, w.dk, w.dv, device=dev)

        def step(dd=d, o=out, st=hT, s=None):
            wr.delta_fwd(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"], o, st,
                         n_h=w.n_h, chunk=w.chunk, stream=s)
        tokens = w.tokens
        kbytes = algorithmic_bytes(w)
        kflops = algorithmic_flops(w)
        kind = "fwd"
        launches = wr.fwd_launches(w.B, w.H, w.T, w.dk, w.dv, w.n_h, w.chunk,
                                   synth.torch_dtype(w.dtype))

    clocks = ClockSampler(dev) if clocks_on else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # ---- device-resident timed region ----
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.region(True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.region(False)
    dist.barrier()
    clock_rec = clocks.stop() if clocks else None
    elapsed = dist.max(t_start.elapsed_time(t_end) / 1e3, dev)
    per_step = [a.elapsed_time(b) / 1e3 for a, b in ev]
    kernel_s = dist.max(sum(per_step) / args.steps, dev)
    ms_per_step = 1e3 * elapsed / args.steps
    value = tokens * dist.world * args.steps / elapsed

    # ---- the two passes of the tensor-core forward timed one by one, through
    #      their own entry points (caller-held T), CUDA events around each ----
    passes = None
    if not decode and launches == 2:
        nt = -(-(w.T * w.n_h) // w.chunk)
        t_mat = torch.empty((w.B, w.H, nt, w.chunk, w.chunk), dtype=torch.bfloat16, device=dev)
        pe = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for _ in range(2):
            wr.delta_ut_transform(d["k"], d["beta"], d["g"], t_mat, n_h=w.n_h, chunk=w.chunk)
            wr.delta_fwd_with_ut(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], t_mat, out,
                                 hT, n_h=w.n_h, chunk=w.chunk)
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            pe[i][0].record(stream)
            wr.delta_ut_transform(d["k"], d["beta"], d["g"], t_mat, n_h=w.n_h, chunk=w.chunk)
            pe[i][1].record(stream)
            wr.delta_fwd_with_ut(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], t_mat, out,
                                 hT, n_h=w.n_h, chunk=w.chunk)
            pe[i][2].record(stream)
        torch.cuda.synchronize(dev)
        ut_s = dist.max(sum(a.elapsed_time(b) for a, b, _ in pe) / 1e3 / args.steps, dev)
        st_s = dist.max(sum(b.elapsed_time(c) for _, b, c in pe) / 1e3 / args.steps, dev)
        e = 2 if w.dtype == "bf16" else 4
        L = w.T * w.n_h
        t_bytes = t_mat.numel() * 2
        ut_bytes = (w.B * L * w.H * (w.dk * e + 4) + (w.B * w.T * w.H * 4 if w.gated else 0)
                    + t_bytes)
        st_bytes = kbytes + t_bytes
        passes = {
            "ut_pass": {"kernel": "ut_kernel", "us": ut_s * 1e6, "share": ut_s / (ut_s + st_s),
                        "bytes_moved": ut_bytes, "gbs": ut_bytes / ut_s / 1e9,
                        "traffic": read_traffic("ut", w.name)},
            "state_pass": {"kernel": "chunk_tc_kernel", "us": st_s * 1e6,
                           "share": st_s / (ut_s + st_s), "bytes_moved": st_bytes,
                           "gbs": st_bytes / st_s / 1e9, "traffic": read_traffic("state", w.name)},
            "extra_bytes_vs_algorithmic": ut_bytes + t_bytes,
        }
        del t_mat

    # ---- end to end through the public API with pinned host buffers:
    #      batch slices on two streams, so that the copies of one slice
    #      overlap the kernels of another ----
    pinned = {n: (None if host[n] is None else host[n].pin_memory()) for n in names}
    h2d = sum(t.numel() * t.element_size() for t in pinned.values() if t is not None)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    if decode:
        d2h = out_h.numel() * out_h.element_size()
        nsl = 1
    else:
        hT_h = torch.empty(hT.shape, dtype=hT.dtype).pin_memory()
        d2h = out_h.numel() * out_h.element_size() + hT_h.numel() * hT_h.element_size()
        nsl = min(w.B, 4)
    streams = [stream, torch.cuda.Stream(dev)]
    bounds = [(i * w.B // nsl, (i + 1) * w.B // nsl) for i in range(nsl)]

    def e2e_step():
        for i, (lo, hi) in enumerate(bounds):
            s = streams[i % 2]
            with torch.cuda.stream(s):
                dd = {n: None if d[n] is None else d[n][lo:hi] for n in names}
                for n in names:
                    if pinned[n] is not None:
                        dd[n].copy_(pinned[n][lo:hi], non_blocking=True)
                if decode:
                    step(s=s)
                    out_h.copy_(out, non_blocking=True)
                else:
                    step(dd, out[lo:hi], hT[lo:hi], s)
                    out_h[lo:hi].copy_(out[lo:hi], non_blocking=True)
                    hT_h[lo:hi].copy_(hT[lo:hi], non_blocking=True)

    def e2e_run(n):
        # the second stream starts after the first's previous work, and the
        # first waits for the second at the end of the step
        for _ in range(n):
            streams[1].wait_stream(streams[0])
            e2e_step()
            streams[0].wait_stream(streams[1])

    e2e_run(min(3, args.warmup))
    torch.cuda.synchronize(dev)
    dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_s = dist.max(e0.elapsed_time(e1) / 1e3, dev)
    e2e_value = tokens * dist.world * args.steps / e2e_s

    # ---- roofline of the step's kernels ----
    hbm = float(peaks["hbm_gbs"])
    achieved = kbytes / kernel_s / 1e9
    t_hbm = kbytes / (hbm * 1e9)
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": read_traffic(kind, w.name),
            "algorithmic_bytes_per_launch": kbytes, "kernel_us": kernel_s * 1e6,
            "kernels_per_step": launches,
            "peak_source": f"hbm_gbs of {peak_src}",
            "spec_peak": SPEC_HBM_GBS, "frac_of_spec_peak": achieved / SPEC_HBM_GBS}
    if passes:
        roof["passes"] = passes
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
    rec = {"workload": w.name, "value": value, "unit": UNIT, "ms_per_step": ms_per_step,
           "step_ms": {k: 1e3 * v for k, v in _spread(per_step).items()},
           "roofline": roof, "config": config_of(w, args),
           "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "slices": nsl, "streams": 2,
                   "host_link_gbs": (h2d + d2h) / (e2e_s / args.steps) / 1e9},
           "clocks": clock_rec, "gpu_launches": launches * args.steps,
           "dtype": "bf16" if w.dtype == "bf16" else "f32"}
    return rec, host


def measure_diagnostics(wr, dev, args):
    """The two diagnostics on the outputs, timed with CUDA events: the
    effective rank of the headline workload's B*H states (128 x 128 float32,
    seeded normal entries) and the attention map of 64-step blocks (B32 H32,
    dk = 128, bf16, gated)."""
    stream = torch.cuda.current_stream(dev)
    w = synth.WORKLOADS[HEADLINE]
    gen = torch.Generator().manual_seed(w.seed + 7)
    states = torch.randn((w.B, w.H, w.dk, w.dv), generator=gen).to(dev)
    mw = synth.WORKLOADS[HEADLINE].with_(name="attention_map_b32_h32_n64_d128_bf16", B=32, H=32, T=64)
    mi = synth.fwd_inputs(mw)
    q, k = mi["q"].to(dev), mi["k"].reshape(mw.B, mw.T, mw.H, mw.dk).to(dev)
    beta, g = mi["beta"].reshape(mw.B, mw.T, mw.H).to(dev), mi["g"].to(dev)
    out = {}
    for name, fn, units, unit in (
            ("effective_rank", lambda: wr.delta_state_erank(states), w.B * w.H, "matrices/s"),
            ("attention_map", lambda: wr.delta_attention_map(q, k, beta, g), mw.B * mw.H, "maps/s")):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for a, b in ev:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
        out[name] = {"us_per_call": us, "value": units / (us * 1e-6), "unit": unit,
                     "units_per_call": units}
    out["effective_rank"]["input"] = f"{w.B}x{w.H} states {w.dk}x{w.dv} float32"
    out["attention_map"]["input"] = f"B{mw.B} H{mw.H} N{mw.T} dk{mw.dk} bf16, gated"
    return out


def measure_prologue(wr, dev, args, peaks):
    """The input prologue on the headline workload's shapes, timed with CUDA
    events: raw q and k ~ N(0, 1) (bf16) and raw beta ~ N(0, 1) through
    SiLU + L2 norm and sigmoid on their own (``delta_prologue``, one pass over
    HBM), and the forward on raw inputs (``delta_fwd_prologue``) beside the
    forward on the same tensors taken as already normalised (``delta_fwd``)."""
    stream = torch.cuda.current_stream(dev)
    w = synth.WORKLOADS[HEADLINE]
    if args.batch:
        w = w.with_(B=args.batch, name=f"{w.name}_batch{args.batch}")
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    gen = torch.Generator(device=dev).manual_seed(w.seed + 11)
    rn = lambda *shape: torch.randn(shape, generator=gen, device=dev)
    q, k, v = (rn(B, T, H, d).to(torch.bfloat16) for d in (dk, dk, dv))
    beta = rn(B, T, H)
    g = torch.sigmoid(rn(B, T, H) * 2.0 + 3.0)
    h0 = rn(B, H, dk, dv) * w.h0_std
    out = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device=dev)
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for a, b in ev:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3

    pro_us = timed(lambda: wr.delta_prologue(q, k, beta))
    fwdp_us = timed(lambda: wr.delta_fwd_prologue(q, k, v, beta, g, h0, out, hT))
    fwd_us = timed(lambda: wr.delta_fwd(q, k, v, beta, g, h0, out, hT))
    nbytes = 2 * (q.numel() * 2 + k.numel() * 2 + beta.numel() * 4)  # read once, write once
    hbm = float(peaks["hbm_gbs"])
    return {"workload": w.name, "input": "raw q, k ~ N(0,1) bf16, raw beta ~ N(0,1), sigmoid",
            "prologue_us": pro_us, "bytes_per_call": nbytes,
            "gbs": nbytes / (pro_us * 1e-6) / 1e9,
            "frac_of_measured_hbm": nbytes / (pro_us * 1e-6) / 1e9 / hbm,
            "fwd_prologue_ms": fwdp_us / 1e3, "fwd_ms": fwd_us / 1e3}


def measure_kda(wr, dev, args, peaks):
    """The channel-wise gate (``delta_fwd_kda``, the CUDA-core kernel) on the
    headline workload's shapes: q, k, v bf16 from the headline recipe (unit
    keys), per-channel alpha = sigmoid(N(0,1) * 2 + 3) float32, timed with CUDA
    events; bytes = the headline's algorithmic bytes + alpha (4 B per key
    channel per token)."""
    stream = torch.cuda.current_stream(dev)
    w = synth.WORKLOADS[HEADLINE]
    if args.batch:
        w = w.with_(B=args.batch, name=f"{w.name}_batch{args.batch}")
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    gen = torch.Generator(device=dev).manual_seed(w.seed + 13)
    rn = lambda *shape: torch.randn(shape, generator=gen, device=dev)
    k = rn(B, T, H, dk)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    q, v = rn(B, T, H, dk).to(torch.bfloat16), rn(B, T, H, dv).to(torch.bfloat16)
    beta = torch.sigmoid(rn(B, T, H))
    alpha = torch.sigmoid(rn(B, T, H, dk) * 2.0 + 3.0)
    h0 = rn(B, H, dk, dv) * w.h0_std
    out = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device=dev)
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    fn = lambda: wr.delta_fwd_kda(q, k, v, beta, alpha, h0, out, hT)
    fn()
    torch.cuda.synchronize(dev)
    steps = max(2, min(args.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    nbytes = algorithmic_bytes(w) + alpha.numel() * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": w.name, "input": "headline shapes, per-channel alpha = sigmoid(2 N(0,1) + 3)",
            "kernel": "chunk_generic_kernel (float32, CUDA cores)", "ms_per_step": ms,
            "value": w.tokens / (ms * 1e-3), "unit": UNIT, "steps": steps,
            "bytes_per_step": nbytes, "gbs": gbs, "frac_of_measured_hbm": gbs / float(peaks["hbm_gbs"])}


def measure_bwd(wr, dev, args, peaks):
    """The gradients (``delta_bwd``, float32 CUDA-core kernel) on the headline
    workload's shapes, timed with CUDA events: q, k, v, dout bf16, beta, g,
    h0 and dhT float32; bytes = every input read once and every gradient
    written once (float32)."""
    stream = torch.cuda.current_stream(dev)
    w = synth.WORKLOADS[HEADLINE]
    if args.batch:
        w = w.with_(B=args.batch, name=f"{w.name}_batch{args.batch}")
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    gen = torch.Generator(device=dev).manual_seed(w.seed + 17)
    rn = lambda *shape: torch.randn(shape, generator=gen, device=dev)
    k = rn(B, T, H, dk)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    q, v, dout = (rn(B, T, H, d).to(torch.bfloat16) for d in (dk, dv, dv))
    beta = torch.sigmoid(rn(B, T, H))
    g = torch.sigmoid(rn(B, T, H) * 2.0 + 3.0)
    h0, dhT = rn(B, H, dk, dv) * w.h0_std, rn(B, H, dk, dv)
    fn = lambda: wr.delta_bwd(q, k, v, beta, g, h0, dout, dhT)
    fn()
    torch.cuda.synchronize(dev)
    steps = 2
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    tok = B * T * H
    nbytes = tok * ((dk * 2 + dv * 2) * 2 + 2 * 4) + 2 * B * H * dk * dv * 4  # inputs
    nbytes += tok * ((dk + dv) * 4 * 2 + 2 * 4) + B * H * dk * dv * 4          # gradients
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": w.name, "kernel": "bwd_kernel (float32, CUDA cores)", "ms_per_step": ms,
            "value": tok / (ms * 1e-3), "unit": UNIT, "steps": steps, "bytes_per_step": nbytes,
            "gbs": gbs, "frac_of_measured_hbm": gbs / float(peaks["hbm_gbs"])}


def run_ours(args, dist):
    import weight_rnn_gb300 as wr

    wr.load_library()
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    peaks, peak_src = load_peaks()
    ids = ORDER if args.workload == "all" else (int(args.workload),)
    recs, hosts = {}, {}
    for wid in ids:
        w = synth.WORKLOADS[wid]
        if args.batch:
            # a smaller copy of the workload (profiler captures): same heads,
            # lengths and distributions, fewer batch rows
            w = w.with_(B=args.batch, name=f"{w.name}_batch{args.batch}")
        recs[wid], host = measure(w, wr, dist, dev, args, peaks, peak_src,
                                  clocks_on=dist.local == 0)
        if wid == ids[0]:
            hosts[wid] = host
        torch.cuda.empty_cache()
    head_id = ids[0]
    head = recs[head_id]
    diagnostics = measure_diagnostics(wr, dev, args) if args.workload == "all" else None
    prologue = measure_prologue(wr, dev, args, peaks) if args.workload == "all" else None
    kda = measure_kda(wr, dev, args, peaks) if args.workload == "all" else None
    bwd = measure_bwd(wr, dev, args, peaks) if args.workload == "all" else None
    w = synth.WORKLOADS[head_id]
    if args.batch:
        w = w.with_(B=args.batch, name=f"{w.name}_batch{args.batch}")

    # ---- CPU oracle on the headline workload (rank 0, N = 1 only) ----
    cpu = None
    if (dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline
            and not w.calls):
        cpu = cpu_baseline(w, hosts[head_id])

    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": head["dtype"], "data": "synthetic",
        "config": head["config"], "roofline": head["roofline"], "cpu_baseline": cpu,
        "e2e": head["e2e"], "clocks": head["clocks"], "step_ms": head["step_ms"],
        "gpu_launches": head["gpu_launches"],
        "gpu": torch.cuda.get_device_name(dev),
        "diagnostics": diagnostics,
        "prologue": prologue,
        "kda": kda,
        "backward": bwd,
        "per_workload": {
            recs[i]["workload"]: {
                "value": recs[i]["value"], "unit": UNIT,
                "ms_per_step": recs[i]["ms_per_step"], "step_ms": recs[i]["step_ms"],
                "roofline_frac": recs[i]["roofline"]["frac"],
                "frac_of_spec_peak": recs[i]["roofline"]["frac_of_spec_peak"],
                "kernel_us": recs[i]["roofline"]["kernel_us"],
                "passes": recs[i]["roofline"].get("passes"),
                "traffic": recs[i]["roofline"]["traffic"],
                "algorithmic_bytes_per_launch":
                    recs[i]["roofline"]["algorithmic_bytes_per_launch"],
                "e2e_value": recs[i]["e2e"]["value"],
                "gpu_launches": recs[i]["gpu_launches"], "clocks": recs[i]["clocks"]}
            for i in ids},
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all", choices=["all", "2", "3", "4", "5"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="run the selected workload(s) with this many batch rows "
                         "instead (for profiler captures; not a bench line)")
    args = ap.parse_args(argv)
    if args.batch < 0:
        ap.error("--batch must be >= 0")
    # at least 3 untimed warm-up steps, whatever is asked
    args.warmup = max(args.warmup, 3)
    dist = Dist()
    if args.impl == "reference":
        return run_reference(args, dist)
    return run_ours(args, dist)


if __name__ == "__main__":
    sys.exit(main())
