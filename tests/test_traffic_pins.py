"""The committed DRAM counters against the code-balance model's bounds on x traffic.

The GPGPU spMVM paper's performance model (arXiv 1112.5588, performance-model section)
charges the right-hand side x by a reuse factor: at best x is read once (n values), at
worst every nonzero reads its own value of x.  On this GPU the worst case is one 32-byte
sector per nonzero.  `profiles/traffic.json` holds, per configuration, the DRAM bytes one
launch of the dominant kernel read (ncu, caches flushed before the launch, so x has to
come from DRAM at least once).  Taking away what the kernel must stream besides x -- every
stored entry's value and column index, and the row length (and, for a sorted layout,
the row number) of every row position -- leaves the bytes spent on x, which must lie
between n values and nnz sectors.  The committed figures are pinned to that model here,
on the CPU; y goes to DRAM as writes, counted apart.
"""
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ROWS = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))

# sizes with a closed form: the 5-point and 7-point Dirichlet stencils lose one
# neighbour per boundary face; the uniform matrix has 16 entries in every row
CLOSED = {
    "lap2d_256": (256 * 256, 5 * 256 * 256 - 4 * 256),
    "lap3d_128": (128 ** 3, 7 * 128 ** 3 - 6 * 128 ** 2),
    "uniform16_16m": (1 << 24, 16 << 24),
}
SECTOR = 32


def _x_bytes(r):
    sv = 8 if r["dtype"] == "f64" else 4
    n_pos = -(-r["n"] // 32) * 32  # row positions, padded to whole slices of 32
    sorted_rows = r["cuda_kernel"].startswith("k_sell_tail")  # the global sort keeps a row number per position
    meta = n_pos * 4 * (2 if sorted_rows else 1)
    return r["dram_bytes_read"] - r["nnz"] * (sv + 4) - meta, sv


def test_every_configuration_has_a_row():
    got = {(r["workload"], r["dtype"]) for r in ROWS}
    assert got == {("lap2d_256", "f64"), ("lap3d_128", "f64"), ("lap3d_128", "f32"), ("hmep_6p2m", "f64"),
                   ("powerlaw_4m", "f64"), ("uniform16_16m", "f32")}


@pytest.mark.parametrize("r", [r for r in ROWS if r["workload"] in CLOSED], ids=lambda r: f"{r['workload']}-{r['dtype']}")
def test_recorded_sizes_match_the_closed_forms(r):
    assert (r["n"], r["nnz"]) == CLOSED[r["workload"]]


@pytest.mark.parametrize("r", ROWS, ids=lambda r: f"{r['workload']}-{r['dtype']}")
def test_x_traffic_within_the_reuse_bounds(r):
    x, sv = _x_bytes(r)
    assert x >= 0.95 * r["n"] * sv, (x, r["n"] * sv)  # x at least once (5 % for the counters' sector rounding)
    assert x <= r["nnz"] * SECTOR, (x, r["nnz"] * SECTOR)
    assert r["dram_bytes_per_launch"] == r["dram_bytes_read"] + r["dram_bytes_write"]


def test_x_reuse_where_the_columns_are_local_or_random():
    """Stencils and the HMEp-shaped matrix read x about once (neighbouring rows share
    their x lines); the uniform random matrix re-reads it, and still no more than once
    per gather."""
    by = {(r["workload"], r["dtype"]): r for r in ROWS}
    for key in (("lap2d_256", "f64"), ("lap3d_128", "f64"), ("lap3d_128", "f32"), ("hmep_6p2m", "f64")):
        x, sv = _x_bytes(by[key])
        assert x <= 1.2 * by[key]["n"] * sv, key
    x, sv = _x_bytes(by[("uniform16_16m", "f32")])
    assert x > 4 * by[("uniform16_16m", "f32")]["n"] * sv
