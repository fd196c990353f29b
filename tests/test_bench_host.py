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
