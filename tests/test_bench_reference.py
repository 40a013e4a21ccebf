"""bench.py --impl reference (the CPU oracle arm) prints the contract's line.

Runs on the CPU: the arm times the oracle on a bounded row sample and never
touches a GPU.
"""
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    t0 = time.time()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "toy",
                        "--steps", "1", "--warmup", "3", "--cpu-seconds", "0.5"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "toy"
    # the timed steps fit in the run: ms_per_step is a step's measured time
    assert d["ms_per_step"] * d["steps"] / 1e3 < time.time() - t0
    # the same config object as the GPU arm (what the workload is)
    sys.path.insert(0, ROOT)
    import bench
    from linear_fp16_gb300 import synth
    assert d["config"] == bench.workload_config(synth.WORKLOADS["toy"], 1)
