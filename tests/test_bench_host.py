"""Host-side logic of bench.py, on the CPU: byte model, rank aggregation (gloo, world size 2),
clock parsing, the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_effective_bytes_formula():
    # 3D Laplacian 128^3 in fp64: nnz*(8+4) + (n+1)*4 + 2*n*8
    n, nnz = 2_097_152, 14_581_760
    assert bench.effective_bytes(n, nnz, 8) == nnz * 12 + (n + 1) * 4 + n * 16 == 216_924_164
    assert bench.effective_bytes(0, 0, 4) == 4


def test_percentile_and_config_selection():
    assert bench.percentile([5.0, 1.0, 3.0], 0.5) == 3.0
    assert bench.percentile([1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0, 8.0, 9.0, 10.0, 11.0], 0.1) == pytest.approx(2.0)
    configs, head = bench.selected_configs("all")
    assert head == ("uniform16_16m", "f32") and head in configs and len(configs) == 6
    assert {c[0] for c in configs} == {"lap2d_256", "lap3d_128", "hmep_6p2m", "powerlaw_4m", "uniform16_16m"}
    assert bench.selected_configs("lap3d_128") == ([("lap3d_128", "f64"), ("lap3d_128", "f32")], ("lap3d_128", "f64"))


def test_region_count_fits_the_timed_budget():
    """11 regions while they fit 30 s of timed work; fewer for long regions, never below 3."""
    assert bench.region_count(1.0) == 11
    assert bench.region_count(2700.0) == 11 and bench.region_count(2800.0) == 10
    assert bench.region_count(5000.0) == 6
    assert bench.region_count(20000.0) == 3 and bench.region_count(1e9) == 3


def test_random_gather_footprint_model():
    """Short rows: one line and one sector per entry.  A long row of sorted columns 0..199
    in float64 (4 values per 32-byte sector, 16 per 128-byte line): six warp instructions
    of 32 entries touch 8 sectors in 2 lines each, the seventh (8 entries) 2 sectors in 1
    line.  The stream adds the matrix, row pointers and y in whole lines and sectors.  The
    bound is the larger of the request time and the sector time."""
    import numpy as np

    from workloads import CSR

    cols = np.concatenate([[5, 900, 4000], np.arange(200)]).astype(np.int32)
    csr = CSR(5000, np.array([0, 3] + [203] * 4999, dtype=np.int32), cols, np.ones(203))
    m = bench.random_gather_footprint(csr)
    assert m["short_row_gathers"] == 3 and m["long_row_sectors"] == 6 * 8 + 2 and m["gather_sectors"] == 53
    assert m["long_row_lines"] == 6 * 2 + 1 and m["gather_lines"] == 16
    stream = 203 * (8 + 4) + 5001 * 4 + 5000 * 8  # 62,440 bytes: 487.8 lines, 1951.25 sectors
    assert m["stream_bytes"] == stream and m["stream_lines"] == 488 and m["stream_sectors"] == 1952
    assert m["lines"] == 16 + 488 and m["sectors"] == 53 + 1952
    m32 = bench.random_gather_footprint(csr.astype(np.float32))  # 8 values per sector, 32 per line
    assert m32["long_row_sectors"] == 6 * 4 + 1 and m32["long_row_lines"] == 6 + 1
    assert bench.gather_bound_ms(m, 504e3, 2005e3 / 2) == pytest.approx(2.0)  # sectors dominate
    assert bench.gather_bound_ms(m, 504e3 / 4, 1e9) == pytest.approx(4.0)  # requests dominate


def test_cpu_leg_parity_field():
    """The CPU leg checks a given y on the rows the oracle computed: the oracle's own
    result (rounded once to double) passes far inside the tolerance; one planted error
    far above the tolerance fails there."""
    import numpy as np

    from workloads import laplacian_2d, uniform_x

    csr = laplacian_2d(40, 30)
    x = uniform_x(csr.n, seed=3)
    import oracle

    y = oracle.spmv(csr, x)["y"]
    rec = bench.cpu_baseline(csr, x, budget_s=0.01, y_gpu=y)
    assert rec["parity"]["within_tolerance"] and rec["parity"]["max_error_ratio"] < 1e-3
    assert rec["parity"]["rows"] == csr.n  # the sample never falls below 20,000 rows (or n)
    bad = y.copy()
    bad[77] += 1e-6
    rec = bench.cpu_baseline(csr, x, budget_s=0.01, y_gpu=bad)
    assert not rec["parity"]["within_tolerance"] and rec["parity"]["worst_row"] == 77
    assert rec["parity"]["max_error_ratio"] > 1.0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist = bench.init_dist(world, "gloo")
    local_seconds = 1.0 + rank  # rank 1 is the slow one
    bench.barrier(world)
    mx = bench.reduce_max(local_seconds, world)
    rate = bench.aggregate_rate(100.0, world, mx)
    out.put((rank, mx, rate))
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]          # every rank sees the slowest time
    assert [r[2] for r in res] == [100.0, 100.0]      # 2 ranks x 100 units / 2 s


def test_clock_summary_parsing():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = [(10.0, "1965, 2070, 800.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"),
                 (10.1, "1980, 2070, 810.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active"),
                 (99.0, "300, 2070, 80.0, 0x0, Not Active, Not Active, Not Active, Not Active")]
    out = s.summary(9.9, 10.2)
    assert out["sm_mhz"] == pytest.approx(1972.5) and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 2


def test_traffic_is_null_when_kernel_changed(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    (tmp_path / "traffic.json").write_text(json.dumps([
        {"workload": "w", "dtype": "f64", "kernel": "sell", "source_sha": "0" * 16, "dram_bytes_per_launch": 5}]))
    assert bench.committed_traffic("w", "f64", "sell") is None
    (tmp_path / "traffic.json").write_text(json.dumps([
        {"workload": "w", "dtype": "f64", "kernel": "sell", "source_sha": bench.source_sha("sell"),
         "dram_bytes_per_launch": 5}]))
    assert bench.committed_traffic("w", "f64", "sell") == 5


def _run_bench(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                          env=env, cwd=ROOT, timeout=300)


def test_reference_arm_prints_one_json_line():
    res = _run_bench(["--impl", "reference", "--workload", "lap2d_small", "--steps", "4", "--warmup", "3"])
    assert res.returncode == 0, res.stderr
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "GFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["steps"] == 4 and line["warmup"] == 3


def test_reference_arm_other_ranks_exit_quietly():
    res = _run_bench(["--impl", "reference", "--workload", "lap2d_small", "--steps", "2", "--warmup", "3"],
                     {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert res.returncode == 0 and res.stdout.strip() == ""
