"""The benchmark's reference arm (the oracle on the host cores) prints the one
JSON line the benchmark contract asks for; runs on the CPU in a few seconds."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(*extra):
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1",
                          *extra], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["vanilla-128e", "deamoe-7b", "suite"])
def test_reference_arm_prints_the_contract_line(workload):
    sys.path.insert(0, ROOT)
    import bench

    d = run_reference("--workload", workload)
    if workload == "suite":
        # the default step: every layer of the five configurations but the tiny one
        assert set(d["config"]["layers"]) == set(bench.SUITE)
        assert all(name in d["config"]["workload"] for name in
                   (bench.WORKLOADS[w].name for w in bench.SUITE))
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 1
    assert d["dtype"] == "f64" and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert isinstance(d["config"]["workload"], str) and d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and isinstance(cb["sample"], str)
    assert cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_our_arm_fails_loudly_without_a_gpu():
    """No GPU: the CUDA arm exits non-zero and prints no result line (there is
    no CPU fallback to report instead)."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    out = subprocess.run([sys.executable, "bench.py", "--steps", "1", "--warmup", "1", "--no-cpu-baseline"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode != 0
    assert not [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
