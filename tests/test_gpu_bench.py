"""bench.py end to end on a GPU: the JSON line carries every key of its
contract, with values that agree with each other, and the benchmarked
histogram matches the oracle bit for bit.

Runs the small uniform workload (1,048,576 keys, 8,192 bins, P = 2) in a
child process, the way the bench is launched.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N, BINS, STEPS = 1_048_576, 8_192, 20


@pytest.fixture(scope="module")
def line():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()   # the child process imports what this builds
    cmd = [sys.executable, "bench.py", "--workload", "uniform-1M-8K", "--steps", str(STEPS),
           "--warmup", "3", "--cpu-seconds", "0.5", "--e2e-steps", "3"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


@pytest.mark.gpu
def test_contract_keys_and_parity(line):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["parity"] == "bit-exact vs oracle"
    assert line["n_gpus"] == 1 and line["steps"] == STEPS and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["vs_baseline"] is None
    cfg = line["config"]
    assert cfg["workload"] == "uniform-1M-8K" and cfg["n"] == N and cfg["num_bins"] == BINS
    assert cfg["cluster_size"] == 2 and "L2-resident" in cfg["l2"]
    # value is whole-job keys per second over the timed steps.
    assert line["value"] == pytest.approx(N / (line["ms_per_step"] / 1e3), rel=1e-6)


@pytest.mark.gpu
def test_roofline_block_is_self_consistent(line):
    r = line["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["kernel"] == "cluster_ship_kernel"
    assert r["algorithmic_bytes"] == 4 * N + 4 * BINS
    assert r["achieved"] == pytest.approx(r["algorithmic_bytes"] / (r["avg_launch_ms"] / 1e3) / 1e9,
                                          rel=1e-6)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-9) and r["frac"] > 0
    lm = r["launch_ms"]
    assert 0 < lm["min"] <= lm["median"] <= lm["max"]
    assert lm["min"] <= r["avg_launch_ms"] <= lm["max"]
    # The cluster kernel is part of the step, never more than all of it.
    assert 0 < r["share_of_step"] <= 1.0 + 1e-6
    # Two launches per step: the cluster kernel and the partial-row reduction.
    assert line["gpu_launches"] == 2 * STEPS


@pytest.mark.gpu
def test_cpu_baseline_and_end_to_end(line):
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] > 0
    assert cpu["unit"] == line["unit"]
    e2e = line["e2e"]
    assert e2e["h2d_bytes_per_step"] == 4 * N and e2e["d2h_bytes_per_step"] == 4 * BINS
    assert e2e["parity"] == "bit-exact vs oracle" and e2e["value"] > 0
    assert e2e["unit"] == line["unit"]


@pytest.mark.gpu
def test_clock_record_is_present(line):
    clocks = line["clocks"]
    assert isinstance(clocks, dict)
    assert "sm_mhz" in clocks and "sm_max_mhz" in clocks and "reasons" in clocks


@pytest.mark.gpu
def test_product_call_is_timed_and_exact(line):
    p = line["product_call"]
    assert p["call"].startswith("dsmem_hist") and p["steps"] >= 1
    assert p["parity"] == "bit-exact vs oracle"
    assert p["value"] == pytest.approx(N / (p["ms_per_step"] / 1e3), rel=1e-6)
    assert p["unit"] == line["unit"] and p["plan"]["cluster_size"] >= 2
