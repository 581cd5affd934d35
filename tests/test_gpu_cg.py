"""Conjugate gradients on the device (spmv_cg) against the CG oracle, on every format.

Tolerances.  The device and the oracle run the same recurrence and differ only in
rounding: each product within 1e-12 * sum |a_ij x_j| per row, each dot product in
its summation order (about n * 2^-53 relative).  Over k <= 12 steps on the 67 x 45
Laplacian (condition number about 1.2e3) these differences grow at most by a factor
of order kappa per step sequence, far below the 1e-9 relative bound used for the
fixed-step comparison.  Converged runs are checked through the true residual, recomputed
with the oracle's product, and by an iteration count within one step of the oracle's
(the stopping decision is the same double comparison on both sides, so only a
residual lying within rounding of the threshold can move it).
"""
import numpy as np
import pytest

import oracle
from oracle.cg import cg as oracle_cg
from tests.cg_bounds import cg_iteration_bound
from tests.gpu_util import build, case_id, torch_cuda
from workloads import integer_x, laplacian_2d, laplacian_3d, make_workload, uniform_x

pytestmark = pytest.mark.gpu

CG_FORMATS = [("auto", {}), ("csr_vector", {}), ("ell_r", {}), ("sell", {"C": 32, "sigma": 1}),
              ("sell", {"C": 64, "sigma": 1 << 30}), ("hyb", {}), ("hyb", {"K": 3, "spill_csr": 0}),
              ("merge", {})]


def true_residual(csr, x, b):
    y = oracle.spmv(csr.astype(np.float64), np.asarray(x, np.float64))["y_hi"]
    b = np.asarray(b, np.float64)
    return np.linalg.norm(b - y) / np.linalg.norm(b)


def device_cg(A, b_np, x0_np=None, **kw):
    torch = torch_cuda()
    b = torch.from_numpy(np.ascontiguousarray(b_np)).cuda()
    x = torch.zeros_like(b) if x0_np is None else torch.from_numpy(np.ascontiguousarray(x0_np)).cuda()
    x, it, res = A.cg(b, x, **kw)
    torch.cuda.synchronize()
    return x.cpu().numpy(), it, res


@pytest.mark.parametrize("fmt,params", CG_FORMATS, ids=[case_id(c) for c in CG_FORMATS])
def test_fixed_steps_match_oracle(fmt, params):
    csr = laplacian_2d(67, 45)
    b = uniform_x(csr.n, seed=11)
    with build(csr, fmt, **params) as A:
        for k in (1, 4, 12):
            x, it, res = device_cg(A, b, rtol=0.0, max_iter=k)
            ref = oracle_cg(csr, b, rtol=0.0, max_iter=k)
            assert it == k == ref["iterations"]
            err = np.max(np.abs(x - ref["x"])) / np.max(np.abs(ref["x"]))
            assert err <= 1e-9, f"{fmt} k={k}: relative difference {err:.3g}"
            assert abs(res - ref["residuals"][-1]) <= 1e-9 * ref["residuals"][-1]


@pytest.mark.parametrize("fmt", ["auto", "merge", "csr_vector"])
def test_converges_like_oracle_fp64(fmt):
    csr, _ = make_workload("lap3d_small")
    b = uniform_x(csr.n, seed=12)
    ref = oracle_cg(csr, b, rtol=1e-8, max_iter=2000)
    with build(csr, fmt) as A:
        x, it, res = device_cg(A, b, rtol=1e-8, max_iter=2000)
    assert abs(it - ref["iterations"]) <= 1, (it, ref["iterations"])
    assert res <= 1e-8
    assert true_residual(csr, x, b) <= 1.01e-8
    assert it <= cg_iteration_bound((37, 29, 23), 1e-8)


def test_converges_fp32():
    csr, _ = make_workload("lap3d_small", dtype=np.float32)
    b = uniform_x(csr.n, seed=13, dtype=np.float32)
    ref = oracle_cg(csr, b, rtol=1e-4, max_iter=2000)
    with build(csr, "auto") as A:
        x, it, res = device_cg(A, b, rtol=1e-4, max_iter=2000)
    assert res <= 1e-4
    # float32 vectors: the recurrence residual may drift from the true one by about
    # u * kappa (6e-8 * 350) relative to ||b||, well inside the 50 % margin
    assert true_residual(csr, x, b) <= 1.5e-4
    assert abs(it - ref["iterations"]) <= max(2, ref["iterations"] // 10)


def test_exact_initial_guess_takes_no_step():
    """b = A x0 with integer x0: the initial residual is exactly zero on both sides."""
    csr = laplacian_2d(67, 45)
    x0 = integer_x(csr.n)
    b = oracle.spmv(csr, x0)["y"]
    with build(csr, "auto") as A:
        x, it, res = device_cg(A, b, x0, rtol=1e-12, max_iter=100)
    assert it == 0 and res == 0.0
    assert np.array_equal(x.view(np.uint64), x0.view(np.uint64))


def test_max_iter_zero_and_zero_rhs():
    csr = laplacian_2d(67, 45)
    b = uniform_x(csr.n, seed=14)
    x0 = uniform_x(csr.n, seed=15)
    ref = oracle_cg(csr, b, x0=x0, max_iter=0)
    with build(csr, "auto") as A:
        x, it, res = device_cg(A, b, x0, rtol=1e-8, max_iter=0)
        assert it == 0 and np.array_equal(x, x0)
        assert abs(res - ref["residuals"][0]) <= 1e-12 * ref["residuals"][0]
        x, it, res = device_cg(A, np.zeros(csr.n), rtol=1e-8, max_iter=50)
        assert it == 0 and res == 0.0 and not x.any()


def test_reproducible_and_stream_independent():
    torch = torch_cuda()
    csr, _ = make_workload("lap3d_small")
    b = uniform_x(csr.n, seed=16)
    with build(csr, "auto") as A:
        x1, it1, _ = device_cg(A, b, rtol=1e-10, max_iter=300)
        s = torch.cuda.Stream()
        bd = torch.from_numpy(b).cuda()
        with torch.cuda.stream(s):
            xd = torch.zeros_like(bd)
            _, it2, _ = A.cg(bd, xd, rtol=1e-10, max_iter=300, stream=s)
        s.synchronize()
        assert it1 == it2
        assert np.array_equal(x1.view(np.uint64), xd.cpu().numpy().view(np.uint64))


def test_indefinite_matrix_reports_breakdown():
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    d = np.array([1.0, -1.0, 2.0, 3.0])
    from workloads import CSR
    csr = CSR(4, np.arange(5, dtype=np.int32), np.arange(4, dtype=np.int32), d)
    with build(csr, "auto") as A:
        b = torch.tensor([1.0, 1.0, 0.0, 0.0], dtype=torch.float64, device="cuda")
        with pytest.raises(spmv.SpmvError) as ei:
            A.cg(b, torch.zeros_like(b), rtol=1e-12, max_iter=10)
        assert ei.value.status == -6  # SPMV_ERR_UNSUPPORTED


def test_invalid_arguments():
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    csr = laplacian_2d(8, 8)
    with build(csr, "auto") as A:
        b = torch.ones(csr.n, dtype=torch.float64, device="cuda")
        for kw in ({"max_iter": -1}, {"rtol": -1.0}, {"rtol": float("nan")}):
            with pytest.raises(spmv.SpmvError) as ei:
                A.cg(b, torch.zeros_like(b), **kw)
            assert ei.value.status == -1
        with pytest.raises(spmv.SpmvError) as ei:
            spmv.spmv_cg(A._h, b, b, 1e-8, 10)  # b and x alias
        assert ei.value.status == -1


def test_full_size_laplacian_3d_128():
    """The 128^3 Laplacian in the headline configuration: the true residual (oracle
    product over every row) meets the tolerance, within the Chebyshev iteration bound."""
    csr, _ = make_workload("lap3d_128")
    b = uniform_x(csr.n, seed=17)
    with build(csr, "auto") as A:
        x, it, res = device_cg(A, b, rtol=1e-6, max_iter=5000)
    assert res <= 1e-6
    assert 0 < it <= cg_iteration_bound((128, 128, 128), 1e-6)
    assert true_residual(csr, x, b) <= 1.05e-6


def test_stop_at_the_first_step_is_exact():
    """A multiple of the identity converges in one step; the host has more iterations
    queued by then, which must neither move x nor count."""
    from workloads import CSR

    n, c = 5000, 4.0
    csr = CSR(n, np.arange(n + 1, dtype=np.int32), np.arange(n, dtype=np.int32), np.full(n, c))
    b = uniform_x(n, seed=51)
    with build(csr, "auto") as A:
        x, it, res = device_cg(A, b, rtol=1e-12, max_iter=1000)
    assert it == 1 and res <= 1e-15
    assert np.max(np.abs(x - b / c)) <= 1e-15 * np.max(np.abs(b / c))


def test_solves_from_two_threads():
    """Two host threads solve on their own handles and streams at the same time: each has
    its own progress record, and each result equals the one-thread result bit for bit."""
    import threading

    torch = torch_cuda()
    csr = laplacian_2d(96, 80)
    cases = [uniform_x(csr.n, seed=61), uniform_x(csr.n, seed=62)]
    ref = []
    for b in cases:
        with build(csr, "auto") as A:
            x, it, _ = device_cg(A, b, rtol=1e-9, max_iter=3000)
            ref.append((x, it))
    out = [None, None]
    errors = []

    def work(i):
        try:
            s = torch.cuda.Stream()
            with build(csr, "auto") as A, torch.cuda.stream(s):
                bd = torch.from_numpy(cases[i]).cuda()
                xd = torch.zeros_like(bd)
                s.synchronize()
                x, it, _ = A.cg(bd, xd, rtol=1e-9, max_iter=3000, stream=s)
                s.synchronize()
                out[i] = (x.cpu().numpy(), it)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    for (x, it), (xr, itr) in zip(out, ref):
        assert it == itr and np.array_equal(x.view(np.uint64), xr.view(np.uint64))
