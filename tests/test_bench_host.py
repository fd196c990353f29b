"""Host-side accounting of bench.py on CPU: the algorithmic bytes behind every
roofline fraction, written out by hand from the per-token sizes of each
workload, and the rule that a DRAM traffic record counts only while the
kernel code it was taken on is unchanged (comments aside)."""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from weight_rnn_gb300 import synth  # noqa: E402

STATE = 128 * 128 * 4  # one float32 state of dk = dv = 128


def test_algorithmic_bytes_deltanet():
    # q, k, v, out: 128 bf16 each; beta float32 -> 1028 B per token; hT per head
    tokens = 8 * 16 * 4096
    assert bench.algorithmic_bytes(synth.WORKLOADS[2]) == tokens * (4 * 256 + 4) + 128 * STATE


def test_algorithmic_bytes_gated_deltanet_with_h0():
    # as above plus the gate (4 B per token); h0 read and hT written per head
    tokens = 4 * 32 * 8192
    assert bench.algorithmic_bytes(synth.WORKLOADS[3]) == tokens * (4 * 256 + 4 + 4) + 2 * 128 * STATE


def test_algorithmic_bytes_gated_deltaproduct():
    # q and out once per token, k, v and beta once per sub-step (n_h = 3), the
    # gate once per token; hT per head, no h0
    tokens = 4 * 16 * 4096
    per_token = 256 + 3 * (256 + 256 + 4) + 256 + 4
    assert per_token == 2064
    assert bench.algorithmic_bytes(synth.WORKLOADS[4]) == tokens * per_token + 64 * STATE


def test_decode_bytes_per_call():
    # float32 q, out once; k, v and beta per sub-step (n_h = 2); the gate; the
    # state read and written once per head
    heads = 256 * 32
    per_head = 512 + 2 * (512 + 512 + 4) + 512 + 4
    assert bench.step_bytes(synth.WORKLOADS[5]) == heads * per_head + 2 * heads * STATE


def test_code_hash_ignores_comments_and_blank_lines():
    a = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    b = "// a header comment\n/* spanning\n   lines */\nint f(int x) {\n\n  return x + 1;\n}\n"
    c = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_traffic_record_needs_the_current_code(monkeypatch):
    name = synth.WORKLOADS[3].name
    recorded = bench.read_traffic("fwd", name)
    if recorded is None:
        # the record is stale for the current sources: nothing to compare
        return
    assert recorded > bench.algorithmic_bytes(synth.WORKLOADS[3]) // 2
    monkeypatch.setattr(bench, "source_sha", lambda kind: "0" * 16)
    assert bench.read_traffic("fwd", name) is None


class FakeNvml:
    """Stands in for the driver's NVML library: answers the read-only queries
    the bench makes, writing through the ctypes references it is given."""

    def __init__(self, mhz=1965, max_mhz=2070, mw=950000, reasons=0x4, init_status=0,
                 new_reason_call=True):
        self.mhz, self.max_mhz, self.mw, self.reasons = mhz, max_mhz, mw, reasons
        self.init_status = init_status
        self.calls = []
        if new_reason_call:
            self.nvmlDeviceGetCurrentClocksEventReasons = self._reasons
        else:
            self.nvmlDeviceGetCurrentClocksThrottleReasons = self._reasons

    def nvmlInit_v2(self):
        return self.init_status

    def nvmlShutdown(self):
        self.calls.append("shutdown")
        return 0

    def nvmlDeviceGetHandleByPciBusId_v2(self, bus, ref):
        self.calls.append(bus)
        ref._obj.value = 1234
        return 0

    def nvmlDeviceGetClockInfo(self, h, kind, ref):
        assert kind == 1  # the SM clock
        ref._obj.value = self.mhz
        return 0

    def nvmlDeviceGetMaxClockInfo(self, h, kind, ref):
        ref._obj.value = self.max_mhz
        return 0

    def nvmlDeviceGetPowerUsage(self, h, ref):
        ref._obj.value = self.mw
        return 0

    def _reasons(self, h, ref):
        ref._obj.value = self.reasons
        return 0


def _poll(lib, before=0.01, inside=0.03):
    import time
    p = bench.NvmlPoller("00000000:01:00.0", lib=lib)
    assert p.ok
    p.start()
    time.sleep(before)
    p.in_region = True
    time.sleep(inside)
    p.in_region = False
    return p.stop()


def test_nvml_poller_counts_samples_inside_the_timed_region():
    lib = FakeNvml()
    rec = _poll(lib)
    assert rec["samples_under_load"] > 0 and rec["samples"] >= rec["samples_under_load"]
    assert rec["sm_mhz"] == 1965 and rec["sm_max_mhz"] == 2070
    assert rec["reasons"] == ["sw_power_cap"]
    assert rec["source"].startswith("nvml")
    assert lib.calls[0] == b"00000000:01:00.0" and lib.calls[-1] == "shutdown"


def test_nvml_poller_names_every_throttle_reason_and_takes_the_older_call():
    rec = _poll(FakeNvml(reasons=0x4 | 0x8 | 0x20 | 0x40 | 0x1, new_reason_call=False))
    assert rec["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap",
                              "sw_thermal_slowdown"]


def test_nvml_poller_reports_failure_instead_of_raising():
    assert not bench.NvmlPoller("00000000:01:00.0", lib=FakeNvml(init_status=1)).ok
    assert not bench.NvmlPoller("00000000:01:00.0", lib=object()).ok
