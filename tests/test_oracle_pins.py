"""Pins for the CSR oracle: it is checked against things other than itself.

* brute force: a dense matrix built from the CSR triples (duplicates summed) times x
  with numpy's matmul, on tiny matrices of every density, with empty and full rows,
  duplicates and unsorted rows;
* exactness on integer-valued inputs;
* special cases: identity (y = x) and permutation matrices (y_i = x_perm(i));
* closed forms of the 1D, 2D and 3D Dirichlet Laplacian stencils applied to
  constant and linear vectors (the 3D_Poisson family of "Development of Krylov
  and AMG linear solvers for large-scale sparse matrices on GPUs");
* a planted-mistake check: oracle builds with a deliberate bug fail these pins.
"""
import os
import tempfile

import numpy as np
import pytest

import oracle
from workloads import (identity, integer_x, laplacian_1d, laplacian_2d, laplacian_3d,
                       permutation_matrix, random_csr, uniform_x)


def dense_of(csr):
    A = np.zeros((csr.n, csr.n), dtype=np.float64)
    rows = np.repeat(np.arange(csr.n), np.diff(csr.row_ptr))
    np.add.at(A, (rows, csr.col_idx.astype(np.int64)), csr.vals.astype(np.float64))
    return A


CASES = [
    dict(n=1, density=1.0),
    dict(n=7, density=0.0),
    dict(n=16, density=0.3, empty_row_fraction=0.3),
    dict(n=33, density=0.1, full_rows=2),
    dict(n=64, density=1.0),
    dict(n=64, density=0.05, duplicates=True),
    dict(n=48, density=0.2, unsorted=True, duplicates=True),
    dict(n=50, density=0.5, empty_row_fraction=0.5, full_rows=3, unsorted=True),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("seed", [11, 12])
def test_matches_dense_gemv(case, seed):
    csr = random_csr(seed=seed, **case)
    x = uniform_x(csr.n, seed=seed + 100)
    ref = oracle.spmv(csr, x)
    y_dense = dense_of(csr) @ x
    # numpy's fp64 sum of <= 64 terms is within 64 ulp of the exact value
    tol = 1e-13 * ref["scale"]
    assert np.all(np.abs(ref["y_hi"] - y_dense) <= tol)


@pytest.mark.parametrize("case", CASES)
def test_integer_inputs_exact(case):
    csr = random_csr(seed=5, integer_values=True, **case)
    x = integer_x(csr.n, seed=9)
    ref = oracle.spmv(csr, x)
    y_dense = dense_of(csr) @ x  # every partial sum is a small integer: exact in fp64
    assert np.array_equal(ref["y"], y_dense)
    assert np.array_equal(ref["y_lo"], np.zeros(csr.n))


def test_float32_values_converted_exactly():
    csr = random_csr(40, 0.3, seed=3, dtype=np.float32, empty_row_fraction=0.2)
    x = uniform_x(40, seed=4, dtype=np.float32)
    ref = oracle.spmv(csr, x)
    # fp32 products are exact in fp64; the dense fp64 sum of <= 40 terms is within 40 ulp(fp64)
    y_dense = dense_of(csr) @ x.astype(np.float64)
    assert np.all(np.abs(ref["y_hi"] - y_dense) <= 1e-13 * np.maximum(ref["scale"], 1e-300))
    assert ref["y"].dtype == np.float32
    # the fp32 result is the long double value rounded once: within half an fp32 ulp
    half_ulp = np.spacing(np.abs(ref["y"])).astype(np.float64) / 2
    assert np.all(np.abs(ref["y"].astype(np.float64) - ref["y_hi"] - ref["y_lo"]) <= half_ulp)


def test_identity_and_permutation_exact():
    n = 1000
    x = uniform_x(n, seed=7)
    assert np.array_equal(oracle.spmv(identity(n), x)["y"], x)
    perm = np.random.default_rng(3).permutation(n)
    assert np.array_equal(oracle.spmv(permutation_matrix(perm), x)["y"], x[perm])


def test_empty_rows_are_positive_zero():
    csr = random_csr(20, 0.2, seed=1, empty_row_fraction=0.5)
    x = uniform_x(20, seed=2) * 0.0 - 0.0  # all -0.0
    y = oracle.spmv(csr, x)["y"]
    assert np.all(y == 0) and not np.any(np.signbit(y))


def test_row_subset_matches_full():
    csr = random_csr(64, 0.2, seed=8)
    x = uniform_x(64, seed=9)
    full = oracle.spmv(csr, x)
    rows = np.array([63, 0, 17, 17, 5])
    sub = oracle.spmv(csr, x, rows=rows)
    for key in ("y", "y_hi", "y_lo", "scale"):
        assert np.array_equal(sub[key], full[key][rows])


def test_rejects_bad_input():
    csr = random_csr(8, 0.5, seed=1)
    bad = type(csr)(csr.n, csr.row_ptr, csr.col_idx.copy(), csr.vals)
    if bad.col_idx.size:
        bad.col_idx[0] = 8
        with pytest.raises(ValueError):
            oracle.spmv(bad, np.zeros(8))


# --------------------------------------------------------------------------- #
# closed forms of the Dirichlet stencils
# --------------------------------------------------------------------------- #


def stencil_closed_form(grid, diag, f):
    """Expected y for a Dirichlet 2d+1-point Laplacian applied to x = f(grid position).

    With all 2d neighbours present y = 0 for a linear f; on the boundary each
    missing neighbour q contributes f(q) evaluated at its virtual position.
    """
    dims = len(grid)
    coords = np.meshgrid(*[np.arange(g) for g in grid], indexing="ij")
    # natural ordering: first coordinate fastest -> transpose to (.., y, x) flattened
    coords = [c.transpose(*reversed(range(dims))).reshape(-1) for c in coords]
    y = np.zeros(coords[0].size)
    for axis in range(dims):
        for step in (-1, 1):
            q = [c.copy() for c in coords]
            q[axis] = q[axis] + step
            missing = (q[axis] < 0) | (q[axis] >= grid[axis])
            y[missing] += f(*q)[missing]
    assert diag == 2 * dims
    return y


@pytest.mark.parametrize("n", [1, 2, 3, 10, 1001])
def test_laplacian_1d_closed_form(n):
    A = laplacian_1d(n)
    c = 3.0
    y = oracle.spmv(A, np.full(n, c))["y"]
    expect = np.zeros(n)
    expect[0] += c
    expect[-1] += c
    if n == 1:
        expect[0] = 2 * c
    assert np.array_equal(y, expect)
    y = oracle.spmv(A, np.arange(n, dtype=np.float64))["y"]
    expect = np.zeros(n)
    expect[0] = -1.0
    expect[-1] += n
    if n == 1:
        expect[0] = 0.0
    assert np.array_equal(y, expect)


@pytest.mark.parametrize("grid", [(256, 256), (5, 3), (1, 9), (17, 31)])
def test_laplacian_2d_closed_form(grid):
    nx, ny = grid
    A = laplacian_2d(nx, ny)
    ix = np.tile(np.arange(nx), ny).astype(np.float64)
    iy = np.repeat(np.arange(ny), nx).astype(np.float64)
    for (a, b, d) in [(0, 0, 2.0), (1, 0, 0), (0, 1, 0), (3, -2, 5)]:
        x = a * ix + b * iy + d
        y = oracle.spmv(A, x)["y"]
        expect = stencil_closed_form((nx, ny), 4, lambda qx, qy: a * qx + b * qy + d)
        assert np.array_equal(y, expect), (a, b, d)


@pytest.mark.parametrize("grid", [(16, 12, 9), (1, 1, 5), (128, 4, 3)])
def test_laplacian_3d_closed_form(grid):
    nx, ny, nz = grid
    A = laplacian_3d(nx, ny, nz)
    n = nx * ny * nz
    idx = np.arange(n)
    ix, iy, iz = idx % nx, (idx // nx) % ny, idx // (nx * ny)
    for (a, b, c, d) in [(0, 0, 0, -1.5), (1, 2, -3, 4)]:
        x = (a * ix + b * iy + c * iz + d).astype(np.float64)
        y = oracle.spmv(A, x)["y"]
        expect = stencil_closed_form((nx, ny, nz), 6, lambda qx, qy, qz: a * qx + b * qy + c * qz + d)
        assert np.array_equal(y, expect), (a, b, c, d)


# --------------------------------------------------------------------------- #
# acceptance rule
# --------------------------------------------------------------------------- #


def test_check_rows_rule():
    csr = random_csr(30, 0.3, seed=4, empty_row_fraction=0.3)
    x = uniform_x(30, seed=5)
    ref = oracle.spmv(csr, x)
    ok, worst, _ = oracle.check_rows(ref["y"], ref, np.float64)
    assert ok and worst <= 1.0
    ok, _, _ = oracle.check_rows(ref["y"], ref, np.float64, exact=True)
    assert ok
    bumped = ref["y"].copy()
    i = int(np.argmax(ref["scale"]))
    bumped[i] += 1e-11 * ref["scale"][i]
    assert not oracle.check_rows(bumped, ref, np.float64)[0]
    empty = np.nonzero(ref["scale"] == 0)[0]
    if empty.size:
        bad = ref["y"].copy()
        bad[empty[0]] = 1e-300
        assert not oracle.check_rows(bad, ref, np.float64)[0]
    nan = ref["y"].copy()
    nan[0] = np.nan
    assert not oracle.check_rows(nan, ref, np.float64)[0]


# --------------------------------------------------------------------------- #
# planted mistakes
# --------------------------------------------------------------------------- #


def _pins_pass(lib):
    """Run a compact version of the pins above against an oracle library."""
    for case in CASES:
        csr = random_csr(seed=11, **case)
        x = uniform_x(csr.n, seed=111)
        ref = oracle.spmv(csr, x, lib=lib)
        y_dense = dense_of(csr) @ x
        if not np.all(np.abs(ref["y_hi"] - y_dense) <= 1e-13 * ref["scale"]):
            return False
    A = laplacian_2d(17, 31)
    ix = np.tile(np.arange(17), 31).astype(np.float64)
    y = oracle.spmv(A, 3 * ix + 5, lib=lib)["y"]
    expect = stencil_closed_form((17, 31), 4, lambda qx, qy: 3 * qx + 5)
    return bool(np.array_equal(y, expect))


def test_pins_pass_on_the_shipped_oracle():
    assert _pins_pass(oracle.load())


@pytest.mark.parametrize("mutation", [1, 2, 3, 4])
def test_pins_catch_planted_mistakes(mutation):
    with tempfile.TemporaryDirectory() as d:
        path = oracle.build(os.path.join(d, f"mut{mutation}.so"), mutation=mutation)
        lib = oracle.load(path)
        assert not _pins_pass(lib), f"mutation {mutation} slipped through the pins"


# --------------------------------------------------------------------------- #
# y = alpha A x + beta y and the multi-vector form
# --------------------------------------------------------------------------- #


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-1.0, 1.0), (2.5, -0.5), (0.0, 3.0), (-3.0, 0.0)])
def test_scaled_matches_dense(alpha, beta):
    csr = random_csr(48, 0.2, seed=21, integer_values=True, duplicates=True, empty_row_fraction=0.2)
    x = integer_x(48, seed=4)
    y_old = integer_x(48, seed=5)
    ref = oracle.spmv_scaled(csr, x, alpha, beta, y_old)
    expect = alpha * (dense_of(csr) @ x) + beta * y_old  # small integers and halves: exact
    assert np.array_equal(ref["y"], expect)
    if alpha == 1.0 and beta == 0.0:
        plain = oracle.spmv(csr, x)
        for key in ("y", "y_hi", "y_lo", "scale"):
            assert np.array_equal(ref[key], plain[key])


def test_scaled_beta_zero_ignores_y():
    csr = random_csr(30, 0.3, seed=2)
    x = uniform_x(30, seed=3)
    y_nan = np.full(30, np.nan)
    ref = oracle.spmv_scaled(csr, x, 2.0, 0.0, y_nan)
    assert np.all(np.isfinite(ref["y"]))
    assert np.all(np.abs(ref["y_hi"] - 2.0 * (dense_of(csr) @ x)) <= 1e-13 * ref["scale"])


@pytest.mark.parametrize("k", [1, 3, 8])
def test_spmm_matches_dense(k):
    csr = random_csr(40, 0.25, seed=7, integer_values=True, empty_row_fraction=0.1)
    rng = np.random.default_rng(k)
    X = rng.integers(-8, 9, size=(40, k)).astype(np.float64)
    Y = rng.integers(-8, 9, size=(40, k)).astype(np.float64)
    ref = oracle.spmm(csr, X, -1.0, 2.0, Y)
    assert ref["y"].shape == (40, k)
    assert np.array_equal(ref["y"], -1.0 * (dense_of(csr) @ X) + 2.0 * Y)


@pytest.mark.parametrize("schedule", ["static", "dynamic"])
@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_openmp_baseline_agrees_with_oracle(schedule, dtype):
    """The multi-core CPU baseline of the bench computes the same product (value-type sums)."""
    from workloads import make_workload
    csr, x = make_workload("powerlaw_small", dtype=dtype)
    y, used = oracle.omp_spmv(csr, x, schedule)
    ok, worst, row = oracle.check_rows(y, oracle.spmv(csr, x), dtype)
    assert ok, (worst, row)
    assert used >= 1
