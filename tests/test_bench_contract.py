"""bench.py's reference arm (the fp64 oracle on the host cores), CPU only.

The reference arm prints the same one-line JSON record as the GPU arm, with
"impl": "reference".  Under torchrun only rank 0 runs it and prints; the other
ranks exit 0 without work.  The toy workload (256 tokens) keeps both runs to
seconds.
"""

import json
import os
import socket
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["bench.py", "--impl", "reference", "--workload", "gqa_toy", "--steps", "2", "--warmup", "1"]


def _json_lines(text):
    return [json.loads(ln) for ln in text.splitlines() if ln.startswith("{")]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_prints_the_contract_line():
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable] + ARGS, cwd=ROOT, capture_output=True, text=True, timeout=300)
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    ln = lines[0]
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in ln, key
    assert ln["impl"] == "reference"
    assert ln["unit"] == "tokens/s" and ln["higher_is_better"] is True and ln["value"] > 0
    assert ln["steps"] == 2
    assert ln["warmup"] == 3  # fewer than three warm-up steps are raised to three
    assert ln["config"]["workload"] == "gqa_toy"
    cb = ln["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == ln["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = ln["e2e"]
    assert e2e["value"] == ln["value"] and e2e["unit"] == ln["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # the line claims only what ran: its timed steps fit in the process's own
    # wall time, and the value is marked as scaled up from the samples
    assert ln["steps"] * ln["ms_per_step"] / 1e3 <= wall
    ex = ln["extrapolation"]
    assert ex["timed_region_s"] <= wall and ex["workload_s_extrapolated"] > 0


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + ARGS
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference"
