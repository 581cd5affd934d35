#!/usr/bin/env python
"""Benchmark of the GB300 SpMV library on every configuration of the metric.

One step = one y = A x (every kernel of the handle's apply plan) over a matrix already
resident in HBM; the format is AUTO, built once before timing (build time is reported
separately).  The five workloads are timed in one run: the 2D Laplacian 256^2 (fp64,
also under a CUDA graph: it fits in L2), the 3D Laplacian 128^3 (fp64 and fp32), the
HMEp-shaped matrix (fp64), the power-law matrix (fp64) and the random uniform matrix
(fp32).  The headline is the largest, the random uniform matrix (16.8 M rows, 268 M
entries); the others are sub-records of the same JSON line, each with its roofline,
its L2-flushed figure and its format.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload all|NAME]

Each configuration: W warm-up applies, then 11 timed regions of K back-to-back applies
(barrier + synchronize around each); value and ms_per_step come from the median region,
with p10/p90 beside them.  GFLOP/s = 2 nnz / t; effective GB/s uses the algorithmic
bytes nnz (value + int32 index) + (n + 1) int32 row pointers + n values of x + n values
of y.  Multi-GPU runs are independent replicas (one process per GPU, no collective on
the data path); ``value`` is the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SpMV GFLOP/s and effective HBM GB/s (fraction of GB300 peak), fp64 & fp32"
UNIT = "GFLOP/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129e6  # replaced by the device's own figure once a GPU is selected (device_l2_bytes)


def device_l2_bytes(torch) -> float:
    """L2 size of the current device in bytes (the GB300 figure if the query fails)."""
    try:
        return float(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except (AttributeError, RuntimeError):
        return L2_BYTES
PROFILE_DIR = os.path.join(ROOT, "profiles")


# --------------------------------------------------------------------------- #
# host-side helpers (also exercised by the CPU tests)
# --------------------------------------------------------------------------- #


def effective_bytes(n: int, nnz: int, value_bytes: int) -> int:
    """Algorithmic bytes of one y = A x: matrix values + int32 indices, int32 row
    pointers, x read once, y written once."""
    return nnz * (value_bytes + 4) + (n + 1) * 4 + 2 * n * value_bytes


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, init_method="env://")
    return dist


def reduce_max(value: float, world: int, device=None) -> float:
    """Maximum of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device_index=None):
    if world <= 1:
        return
    import torch.distributed as dist

    if dist.get_backend() == "nccl" and device_index is not None:
        dist.barrier(device_ids=[device_index])
    else:
        dist.barrier()


def aggregate_rate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: every rank processed units_per_rank in at most max_seconds."""
    return units_per_rank * world / max_seconds


def load_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {"sell": "sell.cu", "ell_r": "sell.cu", "hyb_ell": "sell.cu", "sell+rowsplit": "sell.cu",
                  "ell_r+rowsplit": "sell.cu", "rowsplit_chunks": "sell.cu",
                  "merge_path": "merge.cu", "coo_segmented": "merge.cu", "carry_fixup": "merge.cu"}


def kernel_source(kernel: str) -> str:
    if kernel.startswith("csr_vector"):
        name = "vector.cu"
    elif "_g" in kernel and kernel.split("_g")[-1][:-1].isdigit():  # G threads per row: sell_g4i, ell_r_g8r, ...
        name = "sellg.cu"
    elif kernel.endswith("_v"):  # 16-byte vector loads: sell_v, ell_r_v, hyb_ell_v
        name = "sellv.cu"
    else:
        name = KERNEL_SOURCES.get(kernel, "")
    return os.path.join(ROOT, "sparse_matrix_vector_csr_gb300", "csrc", name)


#: headers every kernel source includes; a change there changes the kernels too
KERNEL_HEADERS = ("spmv_internal.cuh", "device_util.cuh", "sell_common.cuh")


def source_sha(kernel: str) -> str | None:
    """Hash of the source file that holds a kernel and of the shared headers (a committed
    ncu figure is only valid for the kernel it was taken on)."""
    h = hashlib.sha256()
    src = kernel_source(kernel)
    try:
        for path in [src] + [os.path.join(os.path.dirname(src), hd) for hd in KERNEL_HEADERS]:
            with open(path, "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    return h.hexdigest()[:16]


def committed_traffic(workload: str, dtype: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(PROFILE_DIR, "traffic.json")
    try:
        with open(path) as f:
            rows = json.load(f)
    except Exception:
        return None
    for r in rows:
        if r.get("workload") == workload and r.get("dtype") == dtype and r.get("kernel") == kernel:
            if r.get("source_sha") == source_sha(kernel):
                return r.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while a region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []
        self.marks = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if t0 <= ts <= t1] or [p for _, p in rows[-3:]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in inside:
            for name, v in zip(names, p[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(inside[0][1]),
                "reasons": sorted(reasons), "samples": len(inside)}


# --------------------------------------------------------------------------- #
# our arm
# --------------------------------------------------------------------------- #


def _gpu_id(torch):
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


#: every configuration the metric is quoted on, in run order: (workload, value type)
BENCH_CONFIGS = [
    ("lap2d_256", "f64"),
    ("lap3d_128", "f64"),
    ("lap3d_128", "f32"),
    ("hmep_6p2m", "f64"),
    ("powerlaw_4m", "f64"),
    ("uniform16_16m", "f32"),
]
#: the headline: the largest configuration (16.8 M rows, 268 M entries)
HEADLINE = ("uniform16_16m", "f32")
#: timed regions of K applies each; the line reports their median and spread
REPEATS = 11
MIN_REPEATS = 3
TIMED_BUDGET_MS = 30000.0  # timed work per configuration: fewer regions when K applies take long
E2E_BUDGET_S = 10.0  # each of the three end-to-end runs


def region_count(first_region_ms: float) -> int:
    """Timed regions for a configuration whose first region took first_region_ms (max
    over ranks): REPEATS, or as many as fit TIMED_BUDGET_MS, but at least MIN_REPEATS."""
    fit = int(TIMED_BUDGET_MS // max(first_region_ms, 1e-6))
    return max(MIN_REPEATS, min(REPEATS, fit))
#: matrices small enough to sit in L2: timed under a CUDA graph, flagged "not HBM-bound"
GRAPH_TIMED = ("lap2d_256",)
#: applies captured per CUDA graph for the launch-bound configurations
APPLIES_PER_GRAPH = 100
#: gathers of the random-gather probe (about 1 ms on a GB300)
PROBE_GATHERS = 1 << 28


def np_dtype(tag: str):
    import numpy as np

    return np.float64 if tag == "f64" else np.float32


def percentile(values, q):
    v = sorted(values)
    if not v:
        return None
    k = (len(v) - 1) * q
    lo, hi = int(k), min(int(k) + 1, len(v) - 1)
    return v[lo] + (v[hi] - v[lo]) * (k - lo)


def random_gather_footprint(csr, threshold: int = 128) -> dict:
    """Requests (128-byte lines) and sectors (32 bytes) an SM must send to L2 in one apply.
    x gathers: rows of at most `threshold` entries sit in the sliced layout, where a warp
    instruction covers one entry of 32 different rows, so with random columns every such
    gather is a line and a sector of its own; longer rows go to the row-split pass, whose
    warp instruction covers 32 consecutive entries of one row: their distinct lines and
    sectors are counted exactly (columns sorted within a row, so a new line or sector
    starts where col // (values per line or sector) changes).  The stream: the matrix,
    its row pointers and y at their algorithmic size (the B_eff terms other than x), in
    whole lines and sectors -- the least any layout reads and writes."""
    import numpy as np

    lens = np.diff(csr.row_ptr.astype(np.int64))
    sv = csr.vals.dtype.itemsize
    per_sector = 32 // sv
    short = int(lens[lens <= threshold].sum())
    counts = {"long_row_sectors": 0, "long_row_lines": 0}
    for r in np.nonzero(lens > threshold)[0]:
        a, b = int(csr.row_ptr[r]), int(csr.row_ptr[r + 1])
        col = csr.col_idx[a:b].astype(np.int64)
        for key, per in (("long_row_sectors", per_sector), ("long_row_lines", 4 * per_sector)):
            unit = col // per
            new = np.ones(unit.size, dtype=bool)
            new[1:] = unit[1:] != unit[:-1]
            new[::32] = True  # each warp instruction starts afresh (chunks are multiples of 32)
            counts[key] += int(new.sum())
    n, nnz = int(csr.n), int(lens.sum())
    stream = nnz * (sv + 4) + (n + 1) * 4 + n * sv
    g_lines, g_sectors = short + counts["long_row_lines"], short + counts["long_row_sectors"]
    return {"short_row_gathers": short, **counts, "gather_lines": g_lines, "gather_sectors": g_sectors,
            "stream_bytes": stream, "stream_lines": -(-stream // 128), "stream_sectors": -(-stream // 32),
            "lines": g_lines - (-stream // 128), "sectors": g_sectors - (-stream // 32),
            "model": "x gathers: sliced rows one line and one sector per entry, row-split chunks the distinct lines "
                     "and sectors per 32 consecutive entries; stream: matrix, row pointers and y at their "
                     "algorithmic bytes in whole lines and sectors; bound = max(lines / request rate, sectors / "
                     "sector rate)"}


def gather_bound_ms(footprint: dict, line_rate: float, sector_rate: float) -> float:
    """The gather floor of one apply: requests and returned sectors are separate limits."""
    return max(footprint["lines"] / line_rate, footprint["sectors"] / sector_rate) * 1e3


def probe_gather_rate(torch, spmv, x, sectors_per_line: int = 1) -> float:
    """Lane loads (sectors) per second from x (spmv_probe_gather), best of 5 launches."""
    dev = x.device
    out = torch.zeros(1, dtype=torch.float64, device=dev)
    code = 0 if x.dtype == torch.float64 else 1
    stream = torch.cuda.current_stream()
    spmv.spmv_probe_gather(x, x.numel(), code, sectors_per_line, PROBE_GATHERS, out, stream)  # warm-up
    rates = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        done = spmv.spmv_probe_gather(x, x.numel(), code, sectors_per_line, PROBE_GATHERS, out, stream)
        e1.record(stream)
        e1.synchronize()
        rates.append(done / (e0.elapsed_time(e1) / 1e3))
    return max(rates)


def measure_config(torch, spmv, name, tag, steps, warmup, world, dev_index, sampler, peak, peak_kind, keep=False,
                   cpu=False):
    """Build one workload with AUTO, then time REPEATS regions of `steps` back-to-back
    applies (barrier + synchronize on both sides of each), an L2-flushed apply, the
    per-kernel split and, for L2-resident matrices, applies captured in a CUDA graph."""
    import numpy as np

    from workloads import WORKLOADS, make_workload

    t_gen = time.perf_counter()
    csr, x_np = make_workload(name, dtype=np_dtype(tag))
    gen_s = time.perf_counter() - t_gen
    n, nnz, sv = csr.n, csr.nnz, csr.vals.dtype.itemsize
    dev = torch.device("cuda", dev_index)
    rp, ci, vv = (torch.from_numpy(a).to(dev) for a in (csr.row_ptr, csr.col_idx, csr.vals))
    x = torch.from_numpy(x_np).to(dev)
    y = torch.empty_like(x)
    torch.cuda.synchronize()
    t_b = time.perf_counter()
    A = spmv.SpmvMatrix.from_csr(rp, ci, vv)
    build_ms = (time.perf_counter() - t_b) * 1e3
    desc = A.describe()
    stream = torch.cuda.current_stream()
    apply_c = spmv._abi.lib.spmv_apply  # the C entry point, arguments marshalled once
    args = (A._h, x.data_ptr(), y.data_ptr(), stream.cuda_stream or None)
    rc = 0
    for _ in range(warmup):
        rc |= apply_c(*args)
    torch.cuda.synchronize()
    regions, t0, t1 = [], None, None
    n_regions = REPEATS
    while len(regions) < n_regions:
        barrier(world, dev_index)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if t0 is None:
            t0 = time.time()
        e0.record(stream)
        for _ in range(steps):
            rc |= apply_c(*args)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world, dev_index)
        regions.append(e0.elapsed_time(e1))
        if len(regions) == 1:  # every rank takes the same count, from the slowest first region
            n_regions = region_count(reduce_max(regions[0], world, device=dev))
    t1 = time.time()
    if rc:
        raise RuntimeError(f"spmv_apply failed on {name}: {spmv.spmv_last_error_message()}")
    median_ms = statistics.median(regions)
    region_ms = reduce_max(median_ms, world, device=dev)
    # per-kernel split of one apply (separate, event-bracketed launches)
    splits = [A.apply_profiled(x, y) for _ in range(10)]
    per_kernel = [statistics.median(s[i] for s in splits) for i in range(len(splits[0]))]
    # cold: L2 flushed (a write of twice its size) before every apply, outside the events
    flush = torch.empty(int(2 * device_l2_bytes(torch)) // 4, dtype=torch.float32, device=dev)
    cold = []
    for _ in range(15):
        flush.fill_(1.0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        apply_c(*args)
        b.record(stream)
        b.synchronize()
        cold.append(a.elapsed_time(b))
    del flush
    graph_ms = None
    if name in GRAPH_TIMED:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(3):
                apply_c(A._h, x.data_ptr(), y.data_ptr(), s.cuda_stream)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cap = torch.cuda.current_stream().cuda_stream
            for _ in range(APPLIES_PER_GRAPH):
                apply_c(A._h, x.data_ptr(), y.data_ptr(), cap)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = []
        for _ in range(REPEATS):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            reps.append(e0.elapsed_time(e1) / APPLIES_PER_GRAPH)
        graph_ms = statistics.median(reps)
        del g
    gather = None
    if name.startswith(("powerlaw", "uniform")):
        foot = random_gather_footprint(csr)
        line_rate = probe_gather_rate(torch, spmv, x, 1)
        sector_rate = probe_gather_rate(torch, spmv, x, 4)
        bound_ms = gather_bound_ms(foot, line_rate, sector_rate)
        gather = {"probe_gathers_per_s": line_rate, "probe_sectors_per_s": sector_rate, **foot, "bound_ms": bound_ms,
                  "frac_of_gather_bound": bound_ms / (region_ms / steps),
                  "hbm_frac_at_gather_bound": effective_bytes(n, nnz, sv) / (bound_ms / 1e3) / 1e9 / peak,
                  "probe": "spmv_probe_gather on this x, 8 gathers in flight per thread, a full wave of threads, "
                           "best of 5 launches of 2^28 lane loads: random elements (the request rate, one line "
                           "each) and groups of 4 lanes reading the 4 sectors of a random line (the sector rate)"}
    A.close()
    y_host = y.cpu().numpy() if (cpu or keep) else None  # A x, for the parity check of the CPU leg
    del rp, ci, vv, x, y
    torch.cuda.empty_cache()

    beff = effective_bytes(n, nnz, sv)
    kernels = desc["kernels"]
    ms = region_ms / steps
    if len(kernels) == 1:
        kernel_ms = ms
        note = ("single-kernel plan: launch duration = median timed region / steps (consecutive launches "
                "overlap through programmatic dependent launch, so this is the launch-to-launch interval)")
    else:
        dom = max(range(len(per_kernel)), key=lambda i: per_kernel[i])
        kernel_ms = ms * per_kernel[dom] / sum(per_kernel)
        note = f"{kernels[dom]} share {per_kernel[dom] / sum(per_kernel):.3f} of the event-timed apply"
    dom_kernel = kernels[0] if len(kernels) == 1 else kernels[max(range(len(per_kernel)), key=lambda i: per_kernel[i])]
    cold_ms = statistics.median(cold)
    l2 = device_l2_bytes(torch)
    rec = {
        "workload": name, "dtype": tag, "desc": WORKLOADS[name]["desc"], "n": n, "nnz": nnz,
        "value": 2.0 * nnz * world / (ms / 1e3) / 1e9, "unit": UNIT,
        "ms_per_step": ms, "ms_per_step_p10": percentile(regions, 0.1) / steps,
        "ms_per_step_p90": percentile(regions, 0.9) / steps, "regions": len(regions), "steps_per_region": steps,
        "effective_gbs": beff / (ms / 1e3) / 1e9,
        "cold_ms_per_step": cold_ms, "cold_effective_gbs": beff / (cold_ms / 1e3) / 1e9,
        "build_ms": build_ms, "generate_s": gen_s,
        "format": {k: desc[k] for k in ("format", "C", "sigma", "K", "slots", "padded_entries", "n_long_rows",
                                        "segment", "kernels")},
        "per_kernel_ms": per_kernel,
        "l2": ("stream larger than L2: back-to-back applies" if beff > l2 else
               "stream fits in L2: back-to-back figures include L2 reuse; the cold (L2-flushed) figure is the "
               "HBM one"),
        "roofline": {"bound": "hbm", "achieved": beff / (kernel_ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": beff / (kernel_ms / 1e3) / 1e9 / peak,
                     "frac_cold": beff / (cold_ms / 1e3) / 1e9 / peak,
                     "traffic": committed_traffic(name, tag, dom_kernel), "kernel": dom_kernel,
                     "algorithmic_bytes_per_launch": beff, "peak_source": f"{peak_kind} (hbm_gbs)", "note": note},
        "clocks": sampler.summary(t0, t1) if sampler else None,
    }
    if graph_ms is not None:
        rec["graph"] = {"ms_per_step": graph_ms, "applies_per_graph": APPLIES_PER_GRAPH,
                        "value": 2.0 * nnz / (graph_ms / 1e3) / 1e9, "effective_gbs": beff / (graph_ms / 1e3) / 1e9,
                        "frac": beff / (graph_ms / 1e3) / 1e9 / peak,
                        "note": "not HBM-bound: the matrix fits in L2; launch and latency figures"}
    if gather:
        rec["gather_roofline"] = gather
        # the limit that binds here: the requests an SM sends to L2, not HBM bandwidth
        rec["roofline"]["binding_limit"] = {"kind": "L1-to-L2 requests of the x gathers and the stream",
                                            "frac": gather["frac_of_gather_bound"],
                                            "bound_ms": gather["bound_ms"], "see": "gather_roofline"}
    if cpu:  # context per configuration: the oracle on a short row sample, the OpenMP product on all of it
        rec["cpu_oracle"] = cpu_baseline(csr, x_np, budget_s=1.5, y_gpu=y_host)
        rec["cpu_openmp"] = cpu_openmp_baseline(csr, x_np, "dynamic" if name.startswith("powerlaw") else "static")
    if keep:
        rec["_csr"], rec["_x"], rec["_y"] = csr, x_np, y_host
    return rec


def measure_e2e(torch, spmv, csr, x_np, steps):
    """The public host-buffer call (spmv_apply_host) timed by wall clock over `steps`
    calls: every call copies x from page-locked host memory to the device, applies, moves
    y back to page-locked host memory and waits for the stream."""
    dev = torch.device("cuda", torch.cuda.current_device())
    rp, ci, vv = (torch.from_numpy(a).to(dev) for a in (csr.row_ptr, csr.col_idx, csr.vals))
    with spmv.SpmvMatrix.from_csr(rp, ci, vv) as A:
        xt = torch.from_numpy(x_np).pin_memory()
        yt = torch.empty(csr.n, dtype=xt.dtype).pin_memory()
        xh, yh = xt.numpy(), yt.numpy()
        for _ in range(3):
            A.apply_host(xh, yh)
        torch.cuda.synchronize()
        times = []
        for _ in range(3):
            t0 = time.perf_counter()
            for _ in range(steps):
                A.apply_host(xh, yh)
            times.append(time.perf_counter() - t0)
    return statistics.median(times)


def cpu_baseline(csr, x_np, budget_s=10.0, y_gpu=None):
    """The oracle as it stands (single thread, long double) on a row prefix sized to the
    budget.  With y_gpu (the GPU's A x for the same x) the rows the oracle computed are
    also checked against it: the worst |y - y_ref| / (tau * sum |a_ij x_j|) over them."""
    import numpy as np

    import oracle

    probe = min(csr.n, 20000)
    t0 = time.perf_counter()
    oracle.spmv(csr, x_np, rows=np.arange(probe))
    dt = max(time.perf_counter() - t0, 1e-6)
    rows = int(min(csr.n, max(probe, probe * budget_s / dt)))
    t0 = time.perf_counter()
    ref = oracle.spmv(csr, x_np, rows=np.arange(rows))
    dt = time.perf_counter() - t0
    nnz = int(csr.row_ptr[rows])
    out = {"value": 2.0 * nnz / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"rows 0..{rows - 1} of the workload ({nnz} nonzeros), one pass, "
                     f"single-threaded long double (LDBL_MANT_DIG={oracle.ldbl_mant_dig()})",
           "seconds": dt}
    if y_gpu is not None:
        dtype = csr.vals.dtype
        ok, worst, at = oracle.check_rows(np.asarray(y_gpu)[:rows], ref, dtype)
        out["parity"] = {"rows": rows, "within_tolerance": ok, "max_error_ratio": worst, "worst_row": at,
                         "tau": oracle.TAU[np.dtype(dtype)],
                         "rule": "|y - y_ref| <= tau * sum |a_ij x_j| per row (1.0 = at the tolerance)"}
    return out


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform

    return platform.processor() or platform.machine()


def cpu_openmp_baseline(csr, x_np, schedule):
    """The plain OpenMP CSR product (oracle/csr_omp.c) on every host core: median of 11
    applies of the full workload after one warm-up."""
    import oracle

    oracle.omp_spmv(csr, x_np, schedule)
    times = []
    for _ in range(11):
        t0 = time.perf_counter()
        _, used = oracle.omp_spmv(csr, x_np, schedule)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    return {"value": 2.0 * csr.nnz / t / 1e9, "unit": UNIT, "cores": used, "cpu": cpu_model(),
            "kind": "openmp_csr", "schedule": schedule, "ms_per_apply": t * 1e3,
            "sample": "the full workload, median of 11 applies, value-type sums"}


def selected_configs(workload: str):
    """(configs to time, headline) for --workload: all five, or one workload's value types."""
    from workloads import WORKLOADS

    if workload == "all":
        return list(BENCH_CONFIGS), HEADLINE
    picked = [c for c in BENCH_CONFIGS if c[0] == workload]
    if not picked:
        dt = WORKLOADS[workload]["dtype"]
        picked = [(workload, "f64" if dt == __import__("numpy").float64 else "f32")]
    return picked, picked[0]


def run_ours(args):
    import torch

    import sparse_matrix_vector_csr_gb300 as spmv
    from workloads import WORKLOADS

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev_index = torch.cuda.current_device()
    peak, peak_kind = load_peaks()
    configs, headline = selected_configs(args.workload)
    sampler = ClockSampler(_gpu_id(torch)) if rank == 0 else None
    records = {}
    try:
        for name, tag in configs:
            records[(name, tag)] = measure_config(
                torch, spmv, name, tag, args.steps, args.warmup, world, dev_index, sampler, peak, peak_kind,
                keep=(name, tag) == headline,
                cpu=rank == 0 and world == 1 and not args.no_cpu_baseline and (name, tag) != headline)
    finally:
        if sampler:
            sampler.stop()
    head = records[headline]
    csr, x_np, y_host = head.pop("_csr"), head.pop("_x"), head.pop("_y")
    # as many host-buffer calls as fit E2E_BUDGET_S a run (three runs), at least 3: the
    # estimate (the headline apply, max over ranks, plus x in and y out at 150 GB/s) is
    # the same on every rank
    call_s = head["ms_per_step"] / 1e3 + 2.0 * csr.n * csr.vals.dtype.itemsize / 150e9
    e2e_steps = max(3, min(args.steps, int(E2E_BUDGET_S / call_s)))
    e2e_t = reduce_max(measure_e2e(torch, spmv, csr, x_np, e2e_steps), world,
                       device=torch.device("cuda", dev_index))
    if rank != 0:
        return
    sv = csr.vals.dtype.itemsize
    l2_bytes = device_l2_bytes(torch)
    beff = effective_bytes(csr.n, csr.nnz, sv)
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": headline[1], "data": "synthetic",
        "config": {
            "workload": f"{WORKLOADS[headline[0]]['desc']} (nnz={csr.nnz}), {'float64' if sv == 8 else 'float32'}",
            "n": csr.n, "nnz": csr.nnz, "format": head["format"]["format"],
            "parallelism": "replicas" if world > 1 else "single",
            "timing": (f"{head['regions']} timed regions of {args.steps} back-to-back applies after {args.warmup} "
                       "warm-up applies, barrier + synchronize around each region; value and ms_per_step from the "
                       f"median region (max over ranks), p10/p90 beside it; up to {REPEATS} regions, fewer (at least "
                       f"{MIN_REPEATS}) where {REPEATS} would exceed {TIMED_BUDGET_MS / 1e3:.0f} s of timed work"),
            "l2": (f"inputs larger than L2: one apply streams {beff / 1e6:.0f} MB > {l2_bytes / 1e6:.0f} MB L2"
                   if beff > l2_bytes else f"stream of {beff / 1e6:.0f} MB fits in the {l2_bytes / 1e6:.0f} MB L2; "
                                           "cold_* fields flush L2 before every apply"),
            "l2_bytes": int(l2_bytes),
            "configs": [f"{n_}:{t_}" for n_, t_ in configs],
        },
        "ms_per_step_p10": head["ms_per_step_p10"], "ms_per_step_p90": head["ms_per_step_p90"],
        "effective_gbs": head["effective_gbs"],
        "roofline": head["roofline"],
        "gpu_launches": args.steps * len(head["format"]["kernels"]),
        "gpu_launches_note": "kernels of this library launched in one timed region (steps x launches per apply)",
        "e2e": {"value": 2.0 * csr.nnz * e2e_steps * world / e2e_t / 1e9, "unit": UNIT, "steps": e2e_steps,
                "h2d_bytes_per_step": csr.n * sv, "d2h_bytes_per_step": csr.n * sv,
                "note": ("spmv_apply_host on the headline workload: page-locked x -> device, apply, y -> "
                         "page-locked host, stream synchronised every call; median of 3 runs of `steps` calls")},
        "clocks": head["clocks"],
        "headline": {k: v for k, v in head.items() if k not in ("roofline", "clocks")},
        "configs": [{k: v for k, v in records[c].items()} for c in configs if c != headline],
    }
    if "gather_roofline" in head:
        line["gather_roofline"] = head["gather_roofline"]
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(csr, x_np, y_gpu=y_host)
        line["cpu_openmp"] = cpu_openmp_baseline(csr, x_np,
                                                 "dynamic" if headline[0].startswith("powerlaw") else "static")
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- #
# reference arm: the oracle on host cores
# --------------------------------------------------------------------------- #


def run_reference(args):
    import numpy as np

    import oracle
    from workloads import WORKLOADS, make_workload

    rank, world, _ = dist_env()
    if rank != 0:
        return
    _, headline = selected_configs(args.workload)
    csr, x = make_workload(headline[0], dtype=np_dtype(headline[1]))
    total_steps = args.steps + args.warmup
    budget = 90.0
    probe = min(csr.n, 20000)
    t0 = time.perf_counter()
    oracle.spmv(csr, x, rows=np.arange(probe))
    per_row = max(time.perf_counter() - t0, 1e-6) / probe
    rows = int(max(1, min(csr.n, budget / total_steps / per_row)))
    sample = np.arange(rows)
    nnz_s = int(csr.row_ptr[rows])
    for _ in range(args.warmup):
        oracle.spmv(csr, x, rows=sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.spmv(csr, x, rows=sample)
    dt = time.perf_counter() - t0
    value = 2.0 * nnz_s * args.steps / dt / 1e9
    sample_desc = (f"each step: rows 0..{rows - 1} ({nnz_s} nonzeros) of the workload, single-threaded long double "
                   f"oracle (LDBL_MANT_DIG={oracle.ldbl_mant_dig()})")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": headline[1], "data": "synthetic", "impl": "reference",
        "config": {"workload": f"{WORKLOADS[headline[0]]['desc']} (nnz={csr.nnz}), "
                               f"{'float64' if headline[1] == 'f64' else 'float32'}",
                   "n": csr.n, "nnz": csr.nnz},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample_desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


SWEEP_FORMATS = [
    ("auto", {}), ("csr_vector", {}), ("ell_r", {}),
    ("sell", {"C": 32, "sigma": 1}), ("sell", {"C": 64, "sigma": 1}), ("sell", {"C": 32, "sigma": 256}),
    ("sell", {"C": 64, "sigma": 256}), ("sell", {"C": 32, "sigma": 1 << 30}), ("sell", {"C": 64, "sigma": 1 << 30}),
    ("hyb", {}), ("hyb", {"spill_csr": 1}), ("hyb", {"K": 20}), ("merge", {}),
    ("sell", {"row_threads": 1}), ("sell", {"row_threads": 2}), ("sell", {"row_threads": 4}), ("sell", {"row_threads": 8}),
    ("sell", {"row_threads": 16}), ("sell", {"row_threads": 32}), ("sell", {"row_threads": 4, "row_group_mode": 0}),
    ("sell", {"row_threads": 8, "row_group_mode": 0}), ("sell", {"row_threads": 2, "row_group_mode": 2}),
    ("sell", {"row_threads": 4, "row_group_mode": 2}), ("sell", {"row_threads": 8, "row_group_mode": 2}),
    ("ell_r", {"row_threads": 4}), ("sell", {"vector_loads": 1}), ("sell", {"C": 64, "vector_loads": 1}),
    ("sell", {"sigma": 1 << 30, "vector_loads": 1}),
    ("sell", {"staged": 1}), ("sell", {"sigma": 1 << 30, "staged": 1}),
]


def mode_dtypes(args):
    """Value types a single-workload mode runs: --dtypes, else float64 and float32 for the
    Laplacians and the workload's own type for the others."""
    import numpy as np

    if args.dtypes:
        return [np.float64 if t == "f64" else np.float32 for t in args.dtypes.split(",")]
    return [np.float64, np.float32] if args.workload.startswith("lap") else [None]


def run_multi(args):
    """Multi-vector apply Y = A X with k = --nrhs right-hand sides (AUTO format): one JSON line per k."""
    import numpy as np
    import torch

    import sparse_matrix_vector_csr_gb300 as spmv
    from workloads import make_workload

    torch.cuda.set_device(0)
    peak, peak_kind = load_peaks()
    dtypes = mode_dtypes(args)
    for dt in dtypes:
        csr, x_np = make_workload(args.workload, dtype=dt)
        sv = csr.vals.dtype.itemsize
        dev = torch.device("cuda", 0)
        rp, ci, vv = (torch.from_numpy(a).to(dev) for a in (csr.row_ptr, csr.col_idx, csr.vals))
        A = spmv.SpmvMatrix.from_csr(rp, ci, vv, format=args.format)
        for k in sorted({1, args.nrhs}):
            X = torch.rand((csr.n, k), dtype=vv.dtype, device=dev) * 2 - 1
            Y = torch.empty_like(X)
            f = spmv._abi.lib.spmv_apply_multi
            call = (A._h, k, 1.0, X.data_ptr(), k, 0.0, Y.data_ptr(), k, None)
            for _ in range(args.warmup):
                f(*call)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            steps = max(args.steps // 100, 20)
            e0.record()
            for _ in range(steps):
                f(*call)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / steps
            beff = csr.nnz * (sv + 4) + (csr.n + 1) * 4 + 2 * csr.n * sv * k
            print(json.dumps({"workload": args.workload, "dtype": "f64" if sv == 8 else "f32", "nrhs": k,
                              "format": A.describe()["format"], "us_per_apply": ms * 1e3,
                              "gflops": 2.0 * csr.nnz * k / ms / 1e6, "effective_gbs": beff / ms / 1e6,
                              "frac": beff / ms / 1e6 / peak, "peak": f"{peak} GB/s {peak_kind}"}), flush=True)
        A.close()


def run_cg(args):
    """Krylov solver on the device (spmv_cg, or spmv_bicgstab with --solver bicgstab): time
    per iteration from two fixed-step runs, then one solve to 1e-6; one JSON line per value
    type."""
    import numpy as np
    import torch

    import sparse_matrix_vector_csr_gb300 as spmv
    from workloads import make_workload

    torch.cuda.set_device(0)
    peak, peak_kind = load_peaks()
    for dt in (np.float64, np.float32):
        csr, b_np = make_workload(args.workload, dtype=dt)
        sv = csr.vals.dtype.itemsize
        dev = torch.device("cuda", 0)
        rp, ci, vv = (torch.from_numpy(a).to(dev) for a in (csr.row_ptr, csr.col_idx, csr.vals))
        b = torch.from_numpy(b_np).to(dev)
        x = torch.zeros_like(b)
        A = spmv.SpmvMatrix.from_csr(rp, ci, vv, format=args.format)
        if args.solver == "gmres":
            def solve(b_, x_, **kw):
                return A.gmres(b_, x_, restart=args.restart, **kw)
        else:
            solve = A.bicgstab if args.solver == "bicgstab" else A.cg
        solve(b, x, rtol=0.0, max_iter=max(args.warmup, 3))

        def timed(iters):
            x.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            _, it, _ = solve(b, x, rtol=0.0, max_iter=iters)
            e1.record()
            torch.cuda.synchronize()
            assert it == iters
            return e0.elapsed_time(e1)

        long_run, short_run = args.cg, max(args.cg // 4, 1)
        ms_iter = statistics.median((timed(long_run) - timed(short_run)) / (long_run - short_run) for _ in range(5))
        x.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        _, it, res = solve(b, x, rtol=1e-6, max_iter=100000)
        solve_s = time.perf_counter() - t0
        # algorithmic bytes of one iteration.  CG: the product, p.q (2 vectors read), the r
        # update (q, r read; r written), the x and p updates (p, x, r read; x, p written).
        # BiCGSTAB: two products, p update (4 vectors), r_hat.v (2), s (3), t.s and t.t (2),
        # x and r updates with r.r and r_hat.r (5 read, 2 written).
        if args.solver == "bicgstab":
            bytes_iter = 2 * effective_bytes(csr.n, csr.nnz, sv) + 18 * csr.n * sv
            launches = 7
        elif args.solver == "gmres":
            # Arnoldi step j: the product, two Gram-Schmidt passes that each read the j + 1
            # basis vectors twice (dot, then axpy), seven passes over w (dots, axpys with w
            # written, scale); mean j + 1 over a cycle is (m + 1) / 2.  Per cycle, spread over
            # its m steps: x += V y (m vectors, x read and written) and r = b - A x with its norm
            m = args.restart
            beff = effective_bytes(csr.n, csr.nnz, sv)
            bytes_iter = beff + (2 * (m + 1) + 7) * csr.n * sv + ((m + 4) * csr.n * sv + beff) / m
            launches = 6
        else:
            bytes_iter = effective_bytes(csr.n, csr.nnz, sv) + 10 * csr.n * sv
            launches = 4
        print(json.dumps({"workload": args.workload, "dtype": "f64" if sv == 8 else "f32", "solver": args.solver,
                          **({"restart": args.restart} if args.solver == "gmres" else {}),
                          "format": A.describe()["format"], "us_per_iteration": ms_iter * 1e3,
                          "launches_per_iteration": launches, "bytes_per_iteration": bytes_iter,
                          "effective_gbs": bytes_iter / ms_iter / 1e6, "frac": bytes_iter / ms_iter / 1e6 / peak,
                          "peak": f"{peak} GB/s {peak_kind}", "solve_rtol": 1e-6, "solve_iterations": it,
                          "solve_relative_residual": res, "solve_wall_ms": solve_s * 1e3}), flush=True)
        A.close()


def run_orderings(args):
    """The matrix in its given numbering and in the permuted bases (row length, reverse
    Cuthill-McKee): build time (ordering included) and time per apply, one JSON line each."""
    import torch

    import sparse_matrix_vector_csr_gb300 as spmv
    from workloads import make_workload

    torch.cuda.set_device(0)
    peak, peak_kind = load_peaks()
    csr, x_np = make_workload(args.workload)
    sv = csr.vals.dtype.itemsize
    beff = effective_bytes(csr.n, csr.nnz, sv)
    dev = torch.device("cuda", 0)
    rp, ci, vv = (torch.from_numpy(a).to(dev) for a in (csr.row_ptr, csr.col_idx, csr.vals))
    x = torch.from_numpy(x_np).to(dev)
    for ordering in (None, "row_length", "rcm"):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        A = spmv.SpmvMatrix.from_csr(rp, ci, vv, format=args.format, ordering=ordering)
        build_ms = (time.perf_counter() - t0) * 1e3
        xp = A.to_basis(x)
        yp = torch.empty_like(xp)
        apply_c = spmv._abi.lib.spmv_apply
        call = (A._h, xp.data_ptr(), yp.data_ptr(), None)
        for _ in range(args.warmup):
            apply_c(*call)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        steps = max(args.steps // 100, 20)
        e0.record()
        for _ in range(steps):
            apply_c(*call)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        d = A.describe()
        print(json.dumps({"workload": args.workload, "ordering": ordering or "given", "format": d["format"],
                          "kernels": d["kernels"], "build_ms": build_ms, "us_per_apply": ms * 1e3,
                          "effective_gbs": beff / ms / 1e6, "frac": beff / ms / 1e6 / peak,
                          "peak": f"{peak} GB/s {peak_kind}", "slots_per_nnz": d["slots"] / max(csr.nnz, 1)}),
              flush=True)
        A.close()


def run_graph(args):
    """Applies captured in a CUDA graph (R = 100 per graph) against the same applies
    launched one by one: the launch-bound small configurations.  One JSON line per
    value type."""
    import numpy as np
    import torch

    import sparse_matrix_vector_csr_gb300 as spmv
    from workloads import make_workload

    torch.cuda.set_device(0)
    peak, peak_kind = load_peaks()
    dtypes = mode_dtypes(args)
    per_graph = 100
    for dt in dtypes:
        csr, x_np = make_workload(args.workload, dtype=dt)
        sv = csr.vals.dtype.itemsize
        beff = effective_bytes(csr.n, csr.nnz, sv)
        dev = torch.device("cuda", 0)
        rp, ci, vv = (torch.from_numpy(a).to(dev) for a in (csr.row_ptr, csr.col_idx, csr.vals))
        x = torch.from_numpy(x_np).to(dev)
        y = torch.empty_like(x)
        A = spmv.SpmvMatrix.from_csr(rp, ci, vv, format=args.format)
        apply_c = spmv._abi.lib.spmv_apply
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(max(args.warmup, 3)):
                apply_c(A._h, x.data_ptr(), y.data_ptr(), s.cuda_stream)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cap = torch.cuda.current_stream().cuda_stream
            for _ in range(per_graph):
                apply_c(A._h, x.data_ptr(), y.data_ptr(), cap)
        reps = max(args.steps // per_graph, 10)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_graph = e0.elapsed_time(e1) / (reps * per_graph)
        e0.record()
        for _ in range(reps * per_graph):
            apply_c(A._h, x.data_ptr(), y.data_ptr(), None)
        e1.record()
        torch.cuda.synchronize()
        ms_eager = e0.elapsed_time(e1) / (reps * per_graph)
        print(json.dumps({"workload": args.workload, "dtype": "f64" if sv == 8 else "f32",
                          "format": A.describe()["format"], "kernels": A.describe()["kernels"],
                          "applies_per_graph": per_graph, "us_per_apply_graph": ms_graph * 1e3,
                          "us_per_apply_eager": ms_eager * 1e3, "gflops_graph": 2.0 * csr.nnz / ms_graph / 1e6,
                          "effective_gbs_graph": beff / ms_graph / 1e6, "frac_graph": beff / ms_graph / 1e6 / peak,
                          "peak": f"{peak} GB/s {peak_kind}", "bytes_per_apply": beff,
                          "note": "inputs smaller than L2: this measures launch and L2, not HBM"}), flush=True)
        A.close()


def run_sweep(args):
    """One JSON line per storage format on the chosen workload (format comparison)."""
    import numpy as np
    import torch

    import sparse_matrix_vector_csr_gb300 as spmv
    from workloads import WORKLOADS, make_workload

    torch.cuda.set_device(0)
    peak, peak_kind = load_peaks()
    dtypes = mode_dtypes(args)
    for dt in dtypes:
        csr, x_np = make_workload(args.workload, dtype=dt)
        sv = csr.vals.dtype.itemsize
        beff = effective_bytes(csr.n, csr.nnz, sv)
        dev = torch.device("cuda", 0)
        rp, ci, vv = (torch.from_numpy(a).to(dev) for a in (csr.row_ptr, csr.col_idx, csr.vals))
        x = torch.from_numpy(x_np).to(dev)
        y = torch.empty_like(x)
        for fmt, params in SWEEP_FORMATS:
            rec = {"workload": args.workload, "dtype": "f64" if sv == 8 else "f32", "format": fmt, "params": params}
            try:
                A = spmv.SpmvMatrix.from_csr(rp, ci, vv, format=fmt, **params)
            except spmv.SpmvError as e:
                rec["error"] = str(e)
                print(json.dumps(rec), flush=True)
                continue
            apply_c = spmv._abi.lib.spmv_apply
            call = (A._h, x.data_ptr(), y.data_ptr(), None)
            for _ in range(args.warmup):
                apply_c(*call)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            steps = max(args.steps // 100, 20)
            e0.record()
            for _ in range(steps):
                apply_c(*call)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / steps
            d = A.describe()
            rec.update({"chosen": d["format"], "C": d["C"], "sigma": d["sigma"], "K": d["K"],
                        "us_per_apply": ms * 1e3, "gflops": 2.0 * csr.nnz / ms / 1e6,
                        "effective_gbs": beff / ms / 1e6, "frac": beff / ms / 1e6 / peak,
                        "peak": f"{peak} GB/s {peak_kind}", "slots_per_nnz": d["slots"] / max(csr.nnz, 1),
                        "n_long_rows": d["n_long_rows"], "kernels": d["kernels"],
                        "per_kernel_ms": A.apply_profiled(x, y)})
            A.close()
            print(json.dumps(rec), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all",
                    help="all = every configuration (headline: uniform16_16m); or one workload name")
    ap.add_argument("--format", default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dtypes", default="", help="with --sweep / --graph / --nrhs: value types to run, e.g. f64,f32")
    ap.add_argument("--sweep", action="store_true", help="one JSON line per storage format instead of the bench line")
    ap.add_argument("--nrhs", type=int, default=0,
                    help="with --sweep: time the multi-vector apply with this many right-hand sides instead")
    ap.add_argument("--graph", action="store_true",
                    help="time applies captured in a CUDA graph against one-by-one launches (small configurations)")
    ap.add_argument("--orderings", action="store_true",
                    help="time the workload in its given numbering and in the row-length / RCM permuted bases")
    ap.add_argument("--cg", type=int, default=0, metavar="ITERS",
                    help="time the Krylov solver (ITERS fixed steps per run) instead of the bench line")
    ap.add_argument("--solver", choices=["cg", "bicgstab", "gmres"], default="cg", help="with --cg: which solver")
    ap.add_argument("--restart", type=int, default=30, help="with --solver gmres: the restart length m")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    if args.workload == "all" and (args.sweep or args.graph or args.orderings or args.cg > 0):
        args.workload = "lap3d_128"  # the single-workload modes
    if args.impl == "reference":
        run_reference(args)
    elif args.cg > 0:
        run_cg(args)
    elif args.orderings:
        run_orderings(args)
    elif args.graph:
        run_graph(args)
    elif args.sweep and args.nrhs > 0:
        run_multi(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
