"""Pins for the BiCGSTAB oracle (oracle/bicgstab.py): a dense nonsymmetric direct solve,
one step for a multiple of the identity, convergence with the true residual on SPD and
nonsymmetric grid operators, and planted mistakes that must break a pin."""
import numpy as np
import pytest

from oracle.bicgstab import bicgstab
from workloads import CSR, convection_diffusion, laplacian_2d


def dense_to_csr(M):
    n = M.shape[0]
    rows, cols = np.nonzero(M)
    row_ptr = np.zeros(n + 1, np.int32)
    np.add.at(row_ptr, rows + 1, 1)
    return CSR(n, np.cumsum(row_ptr).astype(np.int32), cols.astype(np.int32), M[rows, cols].astype(np.float64))


def dense(csr):
    D = np.zeros((csr.n, csr.n))
    for i in range(csr.n):
        for k in range(csr.row_ptr[i], csr.row_ptr[i + 1]):
            D[i, csr.col_idx[k]] += csr.vals[k]
    return D


def dense_case(mutation=0):
    rng = np.random.default_rng(0)
    n = 30
    A = n * np.eye(n) + rng.standard_normal((n, n)) * 3.0
    b = rng.standard_normal(n)
    out = bicgstab(dense_to_csr(A), b, rtol=1e-13, max_iter=200, _mutation=mutation)
    x_ref = np.linalg.solve(A, b)
    return np.linalg.norm(out["x"] - x_ref) / np.linalg.norm(x_ref), out["iterations"]


def test_dense_nonsymmetric_matches_direct_solve():
    err, it = dense_case()
    assert err <= 1e-10 and 0 < it <= 24  # 18 steps for this system


def test_multiple_of_identity_one_step():
    n, c = 40, 2.5
    A = CSR(n, np.arange(n + 1, dtype=np.int32), np.arange(n, dtype=np.int32), np.full(n, c))
    b = np.random.default_rng(1).standard_normal(n)
    out = bicgstab(A, b, rtol=1e-12, max_iter=10)
    assert out["iterations"] == 1
    assert np.max(np.abs(out["x"] - b / c)) <= 1e-15 * np.max(np.abs(b / c))


@pytest.mark.parametrize("make", [lambda: laplacian_2d(25, 19), lambda: convection_diffusion((13, 11, 7), 0.5),
                                  lambda: convection_diffusion((40, 30), 2.0)])
def test_converges_with_true_residual(make):
    csr = make()
    D = dense(csr)
    b = np.random.default_rng(2).standard_normal(csr.n)
    out = bicgstab(csr, b, rtol=1e-9, max_iter=2000)
    true = np.linalg.norm(b - D @ out["x"]) / np.linalg.norm(b)
    assert out["residuals"][-1] <= 1e-9 and true <= 1.01e-9
    assert np.linalg.norm(out["x"] - np.linalg.solve(D, b)) <= 1e-6 * np.linalg.norm(out["x"])


def test_convection_diffusion_is_nonsymmetric_m_matrix():
    csr = convection_diffusion((6, 5, 4), 0.5)
    D = dense(csr)
    assert not np.allclose(D, D.T)
    off = D - np.diag(np.diag(D))
    assert (off <= 0).all() and (np.diag(D) >= -off.sum(axis=1)).all()


def test_zero_rhs_and_no_steps():
    csr = convection_diffusion((9, 8), 0.5)
    out = bicgstab(csr, np.zeros(csr.n), rtol=1e-8)
    assert out["iterations"] == 0 and not out["x"].any()
    x0 = np.ones(csr.n)
    out = bicgstab(csr, np.ones(csr.n), x0=x0, max_iter=0)
    assert out["iterations"] == 0 and np.array_equal(out["x"], x0)


@pytest.mark.parametrize("mutation", [1, 2, 3])
def test_planted_mistakes_break_a_pin(mutation):
    try:
        err, it = dense_case(mutation)
    except ArithmeticError:
        return
    assert not (err <= 1e-10 and it <= 24)
