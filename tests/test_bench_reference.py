"""The reference arm of bench.py (the fp64 oracle timed on the host cores) on the CPU: its
JSON line carries the contract's keys, the same workload keys as the GPU arm's line, a
cpu_baseline describing the run and an e2e object with no host-device traffic; under
torchrun only rank 0 prints."""

import json
import os
import subprocess
import sys
from pathlib import Path

import bench
from synth import WORKLOADS

ROOT = Path(__file__).resolve().parent.parent
CMD = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_t4", "--steps", "3",
       "--warmup", "1", "--cpu-budget", "1"]


def _run(env_extra):
    env = {**os.environ, **env_extra}
    return subprocess.run(CMD, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_line():
    r = _run({"RANK": "0", "LOCAL_RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] >= 1 and d["ms_per_step"] > 0
    assert d["config"] == bench.workload_config(WORKLOADS["tiny_t4"], 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and "oracle" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_other_ranks_print_nothing():
    r = _run({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
