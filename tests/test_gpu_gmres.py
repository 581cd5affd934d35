"""GMRES(m) on the device (spmv_gmres) against the GMRES oracle.

Tolerances.  The device and the oracle run the same algorithm (Gram-Schmidt twice,
Givens rotations, back-substitution, restarts) and differ only in rounding: each
product within 1e-12 * sum |a_ij x_j| per row, each dot product in another order.
Over a few steps on the 41 x 33 x 19 convection-diffusion operator, and over several
restarts on the small Laplacian, the iterates stay within 1e-9 relative.  Converged
solves are checked through the true residual, recomputed with the oracle's product,
and by an iteration count within two steps of the oracle's: GMRES's residual never
increases, so only a residual within rounding of the threshold can move the stop.
"""
import numpy as np
import pytest

import oracle
from oracle.gmres import gmres as oracle_gmres
from tests.gpu_util import build, case_id, to_device, torch_cuda
from workloads import CSR, make_workload, uniform_x

pytestmark = pytest.mark.gpu

FORMATS = [("auto", {}), ("csr_vector", {}), ("merge", {}), ("hyb", {}), ("sell", {"row_threads": 4}),
           ("sell", {"C": 64, "sigma": 1 << 30})]


def true_residual(csr, x, b):
    y = oracle.spmv(csr.astype(np.float64), np.asarray(x, np.float64))["y_hi"]
    b = np.asarray(b, np.float64)
    return np.linalg.norm(b - y) / max(np.linalg.norm(b), 1e-300)


def device_solve(A, b_np, x0_np=None, **kw):
    torch = torch_cuda()
    b = torch.from_numpy(np.ascontiguousarray(b_np)).cuda()
    x = torch.zeros_like(b) if x0_np is None else torch.from_numpy(np.ascontiguousarray(x0_np)).cuda()
    x, it, res = A.gmres(b, x, **kw)
    torch.cuda.synchronize()
    return x.cpu().numpy(), it, res


@pytest.mark.parametrize("fmt,params", FORMATS, ids=[case_id(c) for c in FORMATS])
def test_fixed_steps_match_oracle(fmt, params):
    csr, _ = make_workload("convdiff_small")
    b = uniform_x(csr.n, seed=81)
    with build(csr, fmt, **params) as A:
        for k in (1, 3, 8):
            x, it, res = device_solve(A, b, restart=30, rtol=0.0, max_iter=k)
            ref = oracle_gmres(csr, b, m=30, rtol=0.0, max_iter=k)
            assert it == k == ref["iterations"]
            err = np.max(np.abs(x - ref["x"])) / np.max(np.abs(ref["x"]))
            assert err <= 1e-9, f"{fmt} k={k}: relative difference {err:.3g}"
            assert abs(res - ref["relative_residual"]) <= 1e-8 * ref["relative_residual"]


def test_restarts_match_oracle():
    csr, _ = make_workload("lap3d_small")
    b = uniform_x(csr.n, seed=82)
    x0 = uniform_x(csr.n, seed=83) * 0.1
    with build(csr, "auto") as A:
        for m, k in ((5, 17), (1, 6), (64, 70)):
            x, it, res = device_solve(A, b, x0, restart=m, rtol=0.0, max_iter=k)
            ref = oracle_gmres(csr, b, x0=x0, m=m, rtol=0.0, max_iter=k)
            assert it == k == ref["iterations"]
            err = np.max(np.abs(x - ref["x"])) / np.max(np.abs(ref["x"]))
            assert err <= 1e-9, f"m={m} k={k}: relative difference {err:.3g}"


@pytest.mark.parametrize("name", ["convdiff_small", "lap3d_small"])
def test_converges_like_oracle(name):
    csr, _ = make_workload(name)
    b = uniform_x(csr.n, seed=84)
    ref = oracle_gmres(csr, b, m=30, rtol=1e-8, max_iter=3000)
    with build(csr, "auto") as A:
        x, it, res = device_solve(A, b, restart=30, rtol=1e-8, max_iter=3000)
    assert res <= 1e-8 and true_residual(csr, x, b) <= 1.01e-8
    assert abs(it - ref["iterations"]) <= 2, (it, ref["iterations"])


def test_converges_fp32():
    csr, _ = make_workload("convdiff_small", dtype=np.float32)
    b = uniform_x(csr.n, seed=85, dtype=np.float32)
    with build(csr, "auto") as A:
        x, it, res = device_solve(A, b, restart=20, rtol=1e-4, max_iter=3000)
    assert res <= 1e-4 and true_residual(csr, x, b) <= 2e-4


def test_three_distinct_eigenvalues_three_steps():
    n = 6000
    d = np.array([1.0, 2.5, 7.0])[np.arange(n) % 3]
    csr = CSR(n, np.arange(n + 1, dtype=np.int32), np.arange(n, dtype=np.int32), d)
    b = uniform_x(n, seed=86)
    with build(csr, "auto") as A:
        x, it, res = device_solve(A, b, restart=10, rtol=1e-12, max_iter=50)
    assert it == 3 and res <= 1e-13
    assert np.max(np.abs(x - b / d)) <= 1e-13 * np.max(np.abs(b / d))


def test_breakdown_zero_rhs_and_errors():
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    n = 500
    zero = CSR(n, np.zeros(n + 1, np.int32), np.zeros(0, np.int32), np.zeros(0))
    with build(zero, "auto") as A:
        b = torch.ones(n, dtype=torch.float64, device="cuda")
        with pytest.raises(spmv.SpmvError) as ei:
            A.gmres(b, torch.zeros_like(b), restart=5, rtol=1e-8, max_iter=20)
        assert ei.value.status == -6
    csr, _ = make_workload("convdiff_small")
    with build(csr, "auto") as A:
        x, it, res = device_solve(A, np.zeros(csr.n), restart=10, rtol=1e-8, max_iter=50)
        assert it == 0 and res == 0.0 and not x.any()
        x, it, _ = device_solve(A, np.ones(csr.n), restart=10, rtol=1e-8, max_iter=0)
        assert it == 0 and not x.any()
        b = torch.ones(csr.n, dtype=torch.float64, device="cuda")
        for bad in (0, 65):
            with pytest.raises(spmv.SpmvError) as ei:
                A.gmres(b, torch.zeros_like(b), restart=bad)
            assert ei.value.status == -1
        with pytest.raises(spmv.SpmvError):
            spmv.spmv_gmres(A._h, b, b[1:], 10, 1e-8, 10)


def test_in_the_permuted_basis():
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    csr, _ = make_workload("convdiff_small")
    b = uniform_x(csr.n, seed=87)
    rp, ci, vv = to_device(csr)
    with spmv.SpmvMatrix.from_csr(rp, ci, vv, ordering="rcm") as A:
        bp = A.to_basis(torch.from_numpy(b).cuda())
        xp, it, res = A.gmres(bp, restart=30, rtol=1e-8, max_iter=3000)
        x = A.from_basis(xp).cpu().numpy()
    assert res <= 1e-8 and true_residual(csr, x, b) <= 1.01e-8


def test_full_size_convection_diffusion_128():
    """The 128^3 upwind convection-diffusion operator: the true residual over every row
    (oracle product) meets the tolerance."""
    csr, _ = make_workload("convdiff3d_128")
    b = uniform_x(csr.n, seed=88)
    with build(csr, "auto") as A:
        x, it, res = device_solve(A, b, restart=30, rtol=1e-6, max_iter=5000)
    assert res <= 1e-6 and 0 < it < 5000
    assert true_residual(csr, x, b) <= 1.01e-6
