"""Pins for the storage-layout definitions in ``oracle.layout``.

* storage counts the GPGPU spMVM paper (arXiv 1112.5588, pJDS section) states:
  constant row length costs N x N_nzr^max in ELLPACK and pJDS alike, and one full
  row plus one entry per other row costs N x N in ELLPACK and (b_r + 1) N - b_r in
  pJDS (``tests/golden/pjds_storage.json``);
* brute force on small inputs: the sorted row order and the slice widths recomputed
  with explicit Python loops;
* the HYB width rule against a brute-force minimisation of its byte model.
"""
import json
import os

import numpy as np
import pytest

from oracle import layout

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pjds_storage.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["one_full_row"])
def test_one_full_row_storage(case):
    N, b_r = case["N"], case["b_r"]
    lens = np.ones(N, dtype=np.int64)
    lens[N // 3] = N
    assert layout.ellpack_entries(lens) == case["ellpack"]
    assert layout.pjds_entries(lens, b_r) == case["pjds"]


@pytest.mark.parametrize("case", _golden()["constant_row_length"])
@pytest.mark.parametrize("C", [32, 64])
@pytest.mark.parametrize("sigma", [1, 256, None])
def test_constant_row_length_has_no_overhead(case, C, sigma):
    N, L = case["N"], case["len"]
    lens = np.full(N, L, dtype=np.int64)
    lay = layout.sell_layout(lens, C, sigma or N)
    assert lay["padded_entries"] == case["entries"]
    assert layout.ellpack_entries(lens) == case["entries"]
    assert np.array_equal(lay["perm"], np.arange(N))


def _brute_order(lens, sigma):
    n = len(lens)
    out = []
    for w0 in range(0, n, sigma):
        idx = list(range(w0, min(n, w0 + sigma)))
        # insertion sort by length, longest first; stable
        res = []
        for i in idx:
            pos = len(res)
            while pos > 0 and lens[res[pos - 1]] < lens[i]:
                pos -= 1
            res.insert(pos, i)
        out.extend(res)
    return np.array(out, dtype=np.int64)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("sigma", [1, 2, 5, 32, 100, 10**9])
def test_sell_order_brute_force(seed, sigma):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 300))
    lens = rng.integers(0, 9, size=n)
    assert np.array_equal(layout.sell_order(lens, sigma), _brute_order(list(lens), min(sigma, n)))


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("C", [1, 4, 32])
def test_sell_widths_brute_force(seed, C):
    rng = np.random.default_rng(seed + 10)
    n = int(rng.integers(1, 200))
    lens = rng.integers(0, 50, size=n)
    sigma = int(rng.integers(1, 64))
    lay = layout.sell_layout(lens, C, sigma)
    order = _brute_order(list(lens), sigma)
    widths, padded, alloc = [], 0, 0
    for s0 in range(0, n, C):
        rows = order[s0:s0 + C]
        w = max(int(lens[r]) for r in rows)
        widths.append(w)
        padded += w * len(rows)
        alloc += w * C
    assert lay["widths"].tolist() == widths
    assert lay["padded_entries"] == padded
    assert lay["allocated_slots"] == alloc
    assert lay["slice_ptr"][0] == 0 and lay["slice_ptr"][-1] == alloc


def test_excluded_rows_count_as_empty():
    lens = np.array([3, 100, 2, 2, 1, 7])
    lay = layout.sell_layout(lens, 2, 6, exclude=[1])
    assert lay["sorted_lens"].tolist() == [7, 3, 2, 2, 1, 0]
    assert lay["perm"].tolist() == [5, 0, 2, 3, 4, 1]


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("value_bytes", [4, 8])
def test_hyb_width_minimises_byte_model(seed, value_bytes):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 3000))
    lens = np.minimum(rng.zipf(1.5 + seed * 0.2, size=n), 400)
    ld = layout.ell_leading_dim(n)
    K = layout.hyb_width(lens, value_bytes, ld)
    costs = [layout.hyb_modeled_bytes(lens, k, value_bytes, ld) for k in range(int(lens.max()) + 1)]
    best = min(costs)
    assert costs[K] == best
    assert all(c > best for c in costs[:K])  # smallest minimiser


def test_hyb_width_cap_and_uniform_rows():
    lens = np.full(1000, 16)
    assert layout.hyb_width(lens, 4) == 16
    assert layout.hyb_width(lens, 4, k_cap=10) == 10
    split = layout.hyb_split(lens, 10)
    assert split["spill_nnz"] == 6000 and split["spill_rows"].size == 1000


@pytest.mark.parametrize("n", [1, 31, 32, 255, 256, 257, 65536])
def test_ell_leading_dimension(n):
    ld = layout.ell_leading_dim(n)
    assert ld >= n and ld % 256 == 0 and ld % 32 == 0 and ld - n < 256
