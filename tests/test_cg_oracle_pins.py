"""Pins for the conjugate-gradient oracle (oracle/cg.py), from the mathematics of CG:
a dense direct solve, one-step convergence on an eigenvector, termination after as
many steps as there are distinct eigenvalues, monotone decrease of the energy norm
of the error, and the Chebyshev iteration bound on Laplacians.  Each planted mistake
must break at least one pin."""
import numpy as np
import pytest

from oracle.cg import cg
from tests.cg_bounds import cg_iteration_bound, laplacian_extreme_eigenvalues
from workloads import CSR, laplacian_1d, laplacian_2d


def dense_to_csr(M):
    n = M.shape[0]
    rows, cols = np.nonzero(M)
    row_ptr = np.zeros(n + 1, np.int32)
    np.add.at(row_ptr, rows + 1, 1)
    return CSR(n, np.cumsum(row_ptr).astype(np.int32), cols.astype(np.int32), M[rows, cols].astype(np.float64))


def csr_to_dense(csr):
    D = np.zeros((csr.n, csr.n))
    for i in range(csr.n):
        for k in range(csr.row_ptr[i], csr.row_ptr[i + 1]):
            D[i, csr.col_idx[k]] += csr.vals[k]
    return D


def spd_case(n=20, seed=0):
    rng = np.random.default_rng(seed)
    M = rng.standard_normal((n, n))
    A = M @ M.T + n * np.eye(n)
    b = rng.standard_normal(n)
    return A, b


def dense_solution_error(mutation=0):
    A, b = spd_case()
    out = cg(dense_to_csr(A), b, rtol=1e-13, max_iter=200, _mutation=mutation)
    x_ref = np.linalg.solve(A, b)
    return np.linalg.norm(out["x"] - x_ref) / np.linalg.norm(x_ref), out["iterations"]


def test_dense_spd_matches_direct_solve():
    err, it = dense_solution_error()
    assert err <= 1e-10
    assert 0 < it <= 20  # at most n steps for an n x n SPD matrix


def test_eigenvector_converges_in_one_step():
    n, k = 50, 3
    i = np.arange(1, n + 1)
    b = np.sin(k * np.pi * i / (n + 1))
    lam = 2.0 - 2.0 * np.cos(k * np.pi / (n + 1))
    out = cg(laplacian_1d(n), b, rtol=1e-10, max_iter=10)
    assert out["iterations"] == 1
    assert np.max(np.abs(out["x"] - b / lam)) <= 1e-12 * np.max(np.abs(b / lam))


def test_three_distinct_eigenvalues_three_steps():
    rng = np.random.default_rng(1)
    d = rng.choice([1.0, 4.0, 9.0], size=30)
    A = np.diag(d)
    b = rng.standard_normal(30)
    out = cg(dense_to_csr(A), b, rtol=1e-12, max_iter=30)
    assert out["iterations"] == 3
    assert np.max(np.abs(out["x"] - b / d)) <= 1e-12


def test_energy_norm_of_error_decreases():
    csr = laplacian_2d(12, 9)
    A = csr_to_dense(csr)
    b = np.random.default_rng(2).standard_normal(csr.n)
    x_star = np.linalg.solve(A, b)
    energies = []
    for k in range(0, 25):
        e = cg(csr, b, rtol=0.0, max_iter=k)["x"] - x_star
        energies.append(float(e @ A @ e))
    assert all(energies[k + 1] < energies[k] for k in range(len(energies) - 1))


def test_recurrence_residual_tracks_true_residual():
    csr = laplacian_2d(20, 20)
    A = csr_to_dense(csr)
    b = np.random.default_rng(3).standard_normal(csr.n)
    out = cg(csr, b, rtol=1e-8, max_iter=1000)
    true = np.linalg.norm(b - A @ out["x"]) / np.linalg.norm(b)
    assert out["residuals"][-1] <= 1e-8 < out["residuals"][-2]
    assert abs(true - out["residuals"][-1]) <= 1e-12
    assert len(out["residuals"]) == out["iterations"] + 1


@pytest.mark.parametrize("dims", [(40,), (30, 30), (12, 10, 9)])
def test_iterations_within_chebyshev_bound(dims):
    from workloads import laplacian_3d
    csr = {1: lambda: laplacian_1d(*dims), 2: lambda: laplacian_2d(*dims), 3: lambda: laplacian_3d(*dims)}[len(dims)]()
    b = np.random.default_rng(4).standard_normal(csr.n)
    out = cg(csr, b, rtol=1e-6, max_iter=5000)
    assert out["residuals"][-1] <= 1e-6
    assert out["iterations"] <= cg_iteration_bound(dims, 1e-6)


def test_laplacian_eigenvalue_closed_form():
    """The extreme eigenvalues used by the bound, against a dense eigensolver."""
    csr = laplacian_2d(7, 5)
    ev = np.linalg.eigvalsh(csr_to_dense(csr))
    lo, hi = laplacian_extreme_eigenvalues((7, 5))
    assert abs(ev[0] - lo) <= 1e-12 and abs(ev[-1] - hi) <= 1e-12


def test_zero_rhs_and_zero_iterations():
    csr = laplacian_2d(6, 6)
    out = cg(csr, np.zeros(csr.n), rtol=1e-8)
    assert out["iterations"] == 0 and not out["x"].any()
    x0 = np.arange(csr.n, dtype=np.float64)
    out = cg(csr, np.ones(csr.n), x0=x0, max_iter=0)
    assert out["iterations"] == 0 and np.array_equal(out["x"], x0)


def test_not_positive_definite_raises():
    A = np.diag([1.0, -1.0, 2.0])
    with pytest.raises(ArithmeticError):
        cg(dense_to_csr(A), np.array([1.0, 1.0, 0.0]), rtol=1e-12)


@pytest.mark.parametrize("mutation", [1, 2, 3])
def test_planted_mistakes_break_a_pin(mutation):
    try:
        err, it = dense_solution_error(mutation)
    except ArithmeticError:
        return  # broke down: caught
    assert not (err <= 1e-10 and it <= 20)
