"""bench.py on a GPU: the JSON line's contract on a small workload (one configuration).

The default run times all five full-size configurations; here one small workload keeps
the test short while every field the line promises is checked: the metric and its
units, the median and spread of the timed regions, the roofline of the dominant kernel
with its peak and fraction, the end-to-end figure with the bytes it moves, the launch
count, the clocks, and the CPU baselines.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         cwd=ROOT, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_contract():
    d = _bench("--workload", "powerlaw_small", "--steps", "10", "--warmup", "3")
    assert d["metric"].startswith("SpMV GFLOP/s") and d["unit"] == "GFLOP/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 10 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["dtype"] == "f64" and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["ms_per_step_p10"] <= d["ms_per_step"] <= d["ms_per_step_p90"]
    nnz = d["config"]["nnz"]
    assert abs(d["value"] - 2.0 * nnz / (d["ms_per_step"] / 1e3) / 1e9) <= 1e-6 * d["value"]
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9 and r["algorithmic_bytes_per_launch"] > 0
    assert d["gpu_launches"] == 10 * len(d["headline"]["format"]["kernels"]) > 0
    e = d["e2e"]
    n = d["config"]["n"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == n * 8 == e["d2h_bytes_per_step"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    par = d["cpu_baseline"]["parity"]  # the GPU result on the rows the oracle computed
    assert par["within_tolerance"] is True and 0 <= par["max_error_ratio"] <= 1.0 and par["rows"] > 0
    assert d["cpu_openmp"]["cores"] >= 1
    g = d["gather_roofline"]  # the power-law shape carries the random-gather roofline
    assert g["probe_gathers_per_s"] > 0 and g["probe_sectors_per_s"] > 0 and 0 < g["frac_of_gather_bound"]
    assert d["roofline"]["binding_limit"]["frac"] == g["frac_of_gather_bound"]
    assert 0 < g["lines"] <= g["sectors"] and g["bound_ms"] == pytest.approx(
        max(g["lines"] / g["probe_gathers_per_s"], g["sectors"] / g["probe_sectors_per_s"]) * 1e3)
    assert d["configs"] == []  # one workload asked for: the headline alone
