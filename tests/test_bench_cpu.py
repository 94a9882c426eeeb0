"""The benchmark's CPU legs: the oracle baselines of every configuration and the reference
arm (`--impl reference`), which times the oracle and prints the JSON contract. They need no
GPU, so they run here on small samples."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("name", sorted(bench.CONFIGS))
def test_config_cpu_baseline(name):
    r = bench.cpu_baseline_config(name, m_sample=128)
    assert r["kind"] == "oracle" and r["unit"] == "TFLOP/s"
    assert r["value"] > 0 and r["cores"] >= 1
    assert r["step_seconds_estimate"] > 0


@pytest.mark.parametrize("workload", ["tensorwise_256", "delayed_step"])
def test_reference_arm_prints_the_contract(workload):
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                          workload, "--steps", "1", "--warmup", "1"], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == bench.CONFIGS[workload]


def test_oracle_quantize_rates_one_and_all_cores():
    """The CPU baseline's quantize leg: the oracle on one core and, in a spawned pool, on all."""
    r = bench.oracle_quantize_rates(rows=64)
    assert r["cores"] >= 1 and r["gbs_1_core"] > 0 and r["gbs_all_cores"] > 0
