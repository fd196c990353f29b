"""Host logic of the multi-rank bench on CPU: two gloo ranks, the barrier
around the timed region, the max-over-ranks of the elapsed time, and the
reference arm running on rank 0 only.  The forward path itself has no
collective (every (b, h) head is an independent sequence), so nothing else is
exchanged between ranks."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, sys.argv[1])
import bench
d = bench.Dist()
d.init("gloo")
d.barrier()
m = d.max(10.0 * d.rank + 0.25)
d.barrier()
print(json.dumps({"rank": d.rank, "world": d.world, "max": m}), flush=True)
d.close()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(code_args, world=2, timeout=120):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                   RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
        procs.append(subprocess.Popen([sys.executable] + code_args, env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=timeout)
            assert p.returncode == 0, err[-2000:]
            outs.append(out)
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    return outs


def test_barrier_and_max_over_ranks():
    outs = _launch(["-c", WORKER, ROOT])
    recs = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(r["rank"] for r in recs) == [0, 1]
    for r in recs:
        assert r["world"] == 2
        assert r["max"] == 10.25        # every rank sees the slowest rank's time


def test_reference_arm_prints_on_rank0_only():
    outs = _launch([os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                    "--steps", "1", "--warmup", "3"], timeout=600)
    lines = [[l for l in o.splitlines() if l.startswith("{")] for o in outs]
    assert len(lines[1]) == 0          # rank 1 exits without work
    assert len(lines[0]) == 1
    rec = json.loads(lines[0][0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
