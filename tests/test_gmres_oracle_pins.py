"""Pins for the GMRES(m) oracle (oracle/gmres.py), each independent of it: the
minimal-residual definition computed by a least-squares solve over an explicit Krylov
basis, the residual estimate against the true residual, a dense nonsymmetric direct
solve within n steps, exactly k steps for a matrix with k distinct eigenvalues,
non-increasing residuals, restarts, and planted mistakes that must break a pin."""
import numpy as np
import pytest

from oracle.gmres import gmres
from workloads import CSR, convection_diffusion, laplacian_2d


def dense_to_csr(M):
    n = M.shape[0]
    rows, cols = np.nonzero(M)
    row_ptr = np.zeros(n + 1, np.int64)
    np.add.at(row_ptr, rows + 1, 1)
    return CSR(n, np.cumsum(row_ptr).astype(np.int32), cols.astype(np.int32), M[rows, cols].astype(np.float64))


def dense(csr):
    D = np.zeros((csr.n, csr.n))
    for i in range(csr.n):
        for k in range(csr.row_ptr[i], csr.row_ptr[i + 1]):
            D[i, csr.col_idx[k]] += csr.vals[k]
    return D


def krylov_minimiser(A, b, x0, k):
    """argmin of ||b - A x|| over x0 + span{r0, A r0, ..., A^(k-1) r0}: an orthonormal
    basis of the Krylov space from numpy's QR, then numpy's least squares."""
    r0 = b - A @ x0
    K = np.empty((A.shape[0], k))
    K[:, 0] = r0 / np.linalg.norm(r0)
    for i in range(1, k):
        K[:, i] = A @ K[:, i - 1]
        K[:, i] /= np.linalg.norm(K[:, i])
    Q, _ = np.linalg.qr(K)
    z = np.linalg.lstsq(A @ Q, r0, rcond=None)[0]
    return x0 + Q @ z


def small_system(seed=0, n=24):
    rng = np.random.default_rng(seed)
    A = n * np.eye(n) + rng.standard_normal((n, n)) * 2.0
    return A, rng.standard_normal(n), rng.standard_normal(n) * 0.1


@pytest.mark.parametrize("k", [1, 2, 3, 5, 8])
def test_iterate_is_the_krylov_minimiser(k):
    A, b, x0 = small_system()
    out = gmres(dense_to_csr(A), b, x0=x0, m=10, rtol=0.0, max_iter=k)
    assert out["iterations"] == k
    ref = krylov_minimiser(A, b, x0, k)
    assert np.linalg.norm(out["x"] - ref) <= 1e-9 * np.linalg.norm(ref)


def test_convection_diffusion_minimiser():
    csr = convection_diffusion((7, 5), 0.5)
    A = dense(csr)
    b = np.random.default_rng(1).standard_normal(csr.n)
    for k in (2, 4, 6):
        out = gmres(csr, b, m=20, rtol=0.0, max_iter=k)
        ref = krylov_minimiser(A, b, np.zeros(csr.n), k)
        assert np.linalg.norm(out["x"] - ref) <= 1e-9 * np.linalg.norm(ref)


def test_estimate_is_the_true_residual():
    """Within a cycle the rotated right-hand side's last entry is the true residual."""
    A, b, x0 = small_system(seed=2)
    for k in (1, 4, 7):
        out = gmres(dense_to_csr(A), b, x0=x0, m=10, rtol=0.0, max_iter=k)
        true = np.linalg.norm(b - A @ out["x"]) / np.linalg.norm(b)
        assert abs(out["estimates"][-1] - true) <= 1e-10 * true + 1e-15


def test_full_gmres_solves_a_dense_system():
    A, b, _ = small_system(seed=3, n=30)
    out = gmres(dense_to_csr(A), b, m=30, rtol=1e-13, max_iter=30)
    ref = np.linalg.solve(A, b)
    assert out["iterations"] <= 30
    assert np.linalg.norm(out["x"] - ref) <= 1e-10 * np.linalg.norm(ref)


def test_three_distinct_eigenvalues_three_steps():
    """The minimal polynomial has degree 3, so the Krylov space is invariant after three
    steps and the third iterate is exact."""
    n = 60
    d = np.array([1.0, 2.5, 7.0])[np.arange(n) % 3]
    csr = CSR(n, np.arange(n + 1, dtype=np.int32), np.arange(n, dtype=np.int32), d)
    b = np.random.default_rng(4).standard_normal(n)
    out = gmres(csr, b, m=10, rtol=1e-12, max_iter=50)
    assert out["iterations"] == 3
    assert np.linalg.norm(out["x"] - b / d) <= 1e-13 * np.linalg.norm(b / d)


def test_residuals_never_increase():
    csr = convection_diffusion((20, 20), 0.5)
    b = np.random.default_rng(5).standard_normal(csr.n)
    out = gmres(csr, b, m=8, rtol=1e-10, max_iter=400)
    est = out["estimates"]
    # within a cycle the estimate cannot grow; across restarts the true residual cannot either
    assert np.all(np.diff(est[:8]) <= 1e-14)
    assert np.all(np.diff(out["residuals"]) <= 1e-14)
    assert out["relative_residual"] <= 1e-10


def test_restart_continues_from_the_cycle_result():
    csr = laplacian_2d(12, 10)
    b = np.random.default_rng(6).standard_normal(csr.n)
    one = gmres(csr, b, m=5, rtol=0.0, max_iter=5)
    two = gmres(csr, b, x0=one["x"], m=5, rtol=0.0, max_iter=5)
    both = gmres(csr, b, m=5, rtol=0.0, max_iter=10)
    assert both["iterations"] == 10
    assert np.array_equal(both["x"], two["x"])


def test_converges_on_grid_operators():
    for csr in (laplacian_2d(30, 25), convection_diffusion((12, 10, 8), 0.5)):
        b = np.random.default_rng(7).standard_normal(csr.n)
        out = gmres(csr, b, m=30, rtol=1e-8, max_iter=3000)
        true = np.linalg.norm(b - dense(csr) @ out["x"]) / np.linalg.norm(b) if csr.n <= 1000 else None
        assert out["relative_residual"] <= 1e-8
        if true is not None:
            assert true <= 1.01e-8


def test_zero_rhs_and_no_steps():
    csr = laplacian_2d(6, 5)
    out = gmres(csr, np.zeros(csr.n), m=5, rtol=1e-8, max_iter=10)
    assert out["iterations"] == 0 and not out["x"].any()
    b = np.ones(csr.n)
    out = gmres(csr, b, m=5, rtol=1e-8, max_iter=0)
    assert out["iterations"] == 0 and not out["x"].any()


def test_singular_operator_breaks_down():
    """A x = b with A = 0 on the Krylov space: the first pivot is zero."""
    n = 5
    csr = CSR(n, np.zeros(n + 1, np.int32), np.zeros(0, np.int32), np.zeros(0))
    with pytest.raises(ArithmeticError):
        gmres(csr, np.ones(n), m=3, rtol=1e-8, max_iter=10)


@pytest.mark.parametrize("mutation", [1, 2, 3])
def test_planted_mistakes_break_a_pin(mutation):
    A, b, x0 = small_system(seed=8)
    csr = dense_to_csr(A)
    broken = False
    for k in (2, 5):
        out = gmres(csr, b, x0=x0, m=10, rtol=0.0, max_iter=k, _mutation=mutation)
        ref = krylov_minimiser(A, b, x0, k)
        true = np.linalg.norm(b - A @ out["x"]) / np.linalg.norm(b)
        if (np.linalg.norm(out["x"] - ref) > 1e-9 * np.linalg.norm(ref)
                or abs(out["estimates"][-1] - true) > 1e-10 * true + 1e-15):
            broken = True
    assert broken
