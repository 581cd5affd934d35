"""Structure checks on the seeded generators (shapes the configs ask for)."""
import numpy as np
import pytest

from workloads import (WORKLOADS, hmep_like, laplacian_2d, laplacian_3d, make_workload, power_law,
                       random_csr, random_uniform_rows)


def _rows_sorted_distinct(csr):
    lens = csr.row_lengths()
    row_of = np.repeat(np.arange(csr.n, dtype=np.int64), lens)
    key = row_of * csr.n + csr.col_idx.astype(np.int64)
    return bool(np.all(key[1:] > key[:-1]))


def test_laplacian_sizes():
    A = laplacian_2d(256, 256)
    assert A.n == 65536 and A.nnz == 5 * 65536 - 4 * 256 == 326656
    B = laplacian_3d(40, 30, 20)
    assert B.nnz == 7 * B.n - 2 * (30 * 20 + 40 * 20 + 40 * 30)
    assert _rows_sorted_distinct(A) and _rows_sorted_distinct(B)
    assert set(np.unique(B.vals).tolist()) == {-1.0, 6.0}


def test_hmep_shape():
    A = hmep_like(n=200_000, block=15_000, seed=3)
    lens = A.row_lengths()
    assert _rows_sorted_distinct(A)
    assert lens.min() >= 1 and lens.max() <= 23
    # every row has its diagonal
    diag_hits = np.zeros(A.n, bool)
    rows = np.repeat(np.arange(A.n), lens)
    diag_hits[rows[A.col_idx == rows]] = True
    assert diag_hits.all()
    # offsets are constant inside a block: rows r and r+1 in the same interior block
    # differ by exactly +1 in every column (contiguous off-diagonals)
    r = 30_001
    a = A.col_idx[A.row_ptr[r]:A.row_ptr[r + 1]]
    b = A.col_idx[A.row_ptr[r + 1]:A.row_ptr[r + 2]]
    if a.size == b.size:
        assert np.array_equal(b - a, np.ones_like(a))


def test_hmep_full_size_row_lengths_statistics():
    # the length distribution is set per 15,000-row block; check it on a block sample
    A = hmep_like(n=2_200_000, block=15_000, seed=3)
    lens = A.row_lengths()
    interior = lens[1_080_000:1_120_000]
    assert interior.min() >= 8 and interior.max() <= 22


def test_power_law_shape():
    A = power_law(n=50_000, zipf_max=2000, n_dense=3, dense_lo=5000, dense_hi=9000, seed=4)
    lens = A.row_lengths()
    dense = A.meta["dense_rows"]
    assert len(dense) == 3
    assert np.all((lens[dense] >= 5000) & (lens[dense] <= 9000))
    others = np.delete(lens, dense)
    assert others.min() >= 1 and others.max() <= 2000
    assert _rows_sorted_distinct(A)


def test_uniform_rows_shape():
    A = random_uniform_rows(n=5000, per_row=16, seed=5)
    assert np.all(A.row_lengths() == 16)
    assert _rows_sorted_distinct(A)
    assert A.vals.dtype == np.float32 and A.vals.min() >= -1 and A.vals.max() < 1


def test_determinism():
    a, xa = make_workload("powerlaw_small")
    b, xb = make_workload("powerlaw_small")
    assert np.array_equal(a.col_idx, b.col_idx) and np.array_equal(a.vals, b.vals)
    assert np.array_equal(xa, xb)


@pytest.mark.parametrize("name", [k for k in WORKLOADS if k.endswith("_small")])
def test_small_workloads_valid(name):
    A, x = make_workload(name)
    assert A.row_ptr[0] == 0 and np.all(np.diff(A.row_ptr) >= 0)
    assert A.col_idx.min() >= 0 and A.col_idx.max() < A.n
    assert x.shape == (A.n,) and x.dtype == A.vals.dtype


def test_random_csr_options():
    A = random_csr(50, 0.3, seed=1, duplicates=True, unsorted=True, empty_row_fraction=0.2, full_rows=2)
    lens = A.row_lengths()
    assert (lens == 50).sum() >= 2 and (lens == 0).sum() >= 1


def test_banded_rows_shape():
    from workloads import banded_random_rows
    csr = banded_random_rows(5000, per_row=40, half_band=100, seed=3)
    lens = np.diff(csr.row_ptr)
    assert (lens == 40).all()
    rows = np.repeat(np.arange(csr.n), lens)
    assert (np.abs(csr.col_idx.astype(np.int64) - rows) <= 100).all()
    c = csr.col_idx.reshape(csr.n, 40)
    assert (np.diff(c, axis=1) > 0).all()  # distinct and sorted inside each row
    assert (np.abs(csr.vals) <= 1).all()


def test_relabelled_laplacian_is_the_same_operator():
    from workloads import laplacian_3d_relabelled
    A = laplacian_3d(7, 5, 4)
    B = laplacian_3d_relabelled(7, 5, 4, seed=1)
    lab = B.meta["labels"]
    DA = np.zeros((A.n, A.n))
    DB = np.zeros((A.n, A.n))
    for r in range(A.n):
        DA[r, A.col_idx[A.row_ptr[r]:A.row_ptr[r + 1]]] = A.vals[A.row_ptr[r]:A.row_ptr[r + 1]]
        DB[r, B.col_idx[B.row_ptr[r]:B.row_ptr[r + 1]]] = B.vals[B.row_ptr[r]:B.row_ptr[r + 1]]
    assert np.array_equal(DB[np.ix_(lab, lab)], DA)  # point p of A is label lab[p] of B
    assert (np.diff(B.col_idx.reshape(-1)[:7]) != 0).all()
