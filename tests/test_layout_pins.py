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


@pytest.mark.parametrize("c", [1.0, 4.0])
@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("value_bytes", [4, 8])
def test_hyb_width_minimises_byte_model(seed, value_bytes, c):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 3000))
    lens = np.minimum(rng.zipf(1.5 + seed * 0.2, size=n), 400)
    ld = layout.ell_leading_dim(n)
    K = layout.hyb_width(lens, value_bytes, ld, c=c)
    costs = [layout.hyb_modeled_bytes(lens, k, value_bytes, ld, c=c) for k in range(int(lens.max()) + 1)]
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


# --------------------------------------------------------------------------- #
# slot placement: column-major and column-grouped (interleaved) layouts
# --------------------------------------------------------------------------- #


@pytest.mark.parametrize("stride,width,group", [(32, 12, 4), (64, 16, 8), (32, 32, 32), (40, 6, 2), (32, 7, 1)])
def test_interleaved_offsets_enumerate_groups_rows_lanes(stride, width, group):
    """Walking the slice group of columns by group, then row by row, then column by column
    visits offsets 0, 1, 2, ... -- the column-grouped layout's definition."""
    width = -(-width // group) * group
    for interleaved in (True, False):
        for (q, j), off in _walk_offsets(stride, width, group, interleaved).items():
            assert layout.slot_offset(q, j, stride, group, interleaved) == off


@pytest.mark.parametrize("group", [2, 4, 8, 16, 32])
def test_interleaved_warp_reads_consecutive_slots(group):
    """32 threads = 32/group rows x group lanes; at step k lane l of row q reads entry
    k*group + l: the warp's 32 offsets are 32 consecutive slots."""
    stride = 64
    for q0 in range(0, stride, 32 // group):
        for k in range(3):
            offs = sorted(int(layout.slot_offset(q0 + r, k * group + l, stride, group, True))
                          for r in range(32 // group) for l in range(group))
            assert offs == list(range(offs[0], offs[0] + 32))


def _walk_offsets(stride, width, group, interleaved):
    """Offsets of (q, j) by walking the slice in the layout's order (no formula)."""
    order = {}
    if interleaved:
        walk = ((q, jg * group + lane) for jg in range(width // group) for q in range(stride) for lane in range(group))
    else:
        walk = ((q, j) for j in range(width) for q in range(stride))
    for k, key in enumerate(walk):
        order[key] = k
    return order


def _brute_slots(csr, C, sigma, exclude, group, interleaved, ell_ld=None):
    lens = layout.row_lengths(csr.row_ptr)
    round_to = group if interleaved else 1
    if ell_ld is None:
        lay = layout.sell_layout(lens, C, sigma, exclude=exclude, group=round_to)
        col = np.zeros(int(lay["slice_ptr"][-1]), np.int32)
        val = np.zeros(col.size, csr.vals.dtype)
        walks = [_walk_offsets(C, int(w), group, interleaved) for w in lay["widths"]]
        for p, r in enumerate(lay["perm"]):
            s, q = divmod(p, C)
            for j in range(int(lay["sorted_lens"][p])):
                off = walks[s][(q, j)]
                col[lay["slice_ptr"][s] + off] = csr.col_idx[csr.row_ptr[r] + j]
                val[lay["slice_ptr"][s] + off] = csr.vals[csr.row_ptr[r] + j]
        return col, val
    stored = lens.copy()
    if exclude is not None:
        stored[exclude] = 0
    w = -(-int(stored.max()) // round_to) * round_to
    col = np.zeros(ell_ld * w, np.int32)
    val = np.zeros(col.size, csr.vals.dtype)
    walk = _walk_offsets(ell_ld, w, group, interleaved)
    for r in range(csr.n):
        for j in range(int(stored[r])):
            off = walk[(r, j)]
            col[off] = csr.col_idx[csr.row_ptr[r] + j]
            val[off] = csr.vals[csr.row_ptr[r] + j]
    return col, val


@pytest.mark.parametrize("C,sigma,group,interleaved", [(32, 1, 1, False), (32, 8, 4, True), (64, 1000, 8, True),
                                                       (32, 1, 2, False), (32, 16, 32, True), (64, 1, 8, False)])
def test_sell_slots_brute_force(C, sigma, group, interleaved):
    from workloads import random_csr
    csr = random_csr(150, density=0.08, seed=7)
    lens = layout.row_lengths(csr.row_ptr)
    exclude = layout.long_rows(lens, 20)
    got = layout.sell_slots(csr, C, sigma, exclude=exclude, group=group, interleaved=interleaved)
    exp = _brute_slots(csr, C, sigma, exclude, group, interleaved)
    assert np.array_equal(got[0], exp[0]) and np.array_equal(got[1], exp[1])


@pytest.mark.parametrize("group,interleaved", [(1, False), (4, True), (8, False)])
def test_ell_slots_brute_force(group, interleaved):
    from workloads import random_csr
    csr = random_csr(90, density=0.1, seed=8)
    got = layout.sell_slots(csr, 0, 1, group=group, interleaved=interleaved, ell_ld=96)
    exp = _brute_slots(csr, 0, 1, None, group, interleaved, ell_ld=96)
    assert np.array_equal(got[0], exp[0]) and np.array_equal(got[1], exp[1])


@pytest.mark.parametrize("C,gval", [(32, 2), (64, 4)])
def test_vector_layout_slots_brute_force(C, gval):
    """The 16-byte vector layout: indices in groups of 4, values in groups of gval (2
    doubles or 4 floats), slice widths rounded to a multiple of 4."""
    from workloads import random_csr
    csr = random_csr(140, density=0.07, seed=9)
    lens = layout.row_lengths(csr.row_ptr)
    got = layout.sell_slots(csr, C, 1, group=4, interleaved=True, group_val=gval, round_to=4)
    lay = layout.sell_layout(lens, C, 1, group=4)
    col = np.zeros(int(lay["slice_ptr"][-1]), np.int32)
    val = np.zeros(col.size, csr.vals.dtype)
    for p_, r in enumerate(lay["perm"]):
        s_, q = divmod(p_, C)
        wc = _walk_offsets(C, int(lay["widths"][s_]), 4, True)
        wv = _walk_offsets(C, int(lay["widths"][s_]), gval, True)
        for j in range(int(lay["sorted_lens"][p_])):
            col[lay["slice_ptr"][s_] + wc[(q, j)]] = csr.col_idx[csr.row_ptr[r] + j]
            val[lay["slice_ptr"][s_] + wv[(q, j)]] = csr.vals[csr.row_ptr[r] + j]
    assert np.array_equal(got[0], col) and np.array_equal(got[1], val)

