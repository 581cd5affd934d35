"""Device allocation failures, injected on the host, and the memory they must not leak.

SPMV_FAIL_ALLOC=k makes the library's k-th device allocation (counted from when the
variable took that value) fail as if the device were out of memory.  Each test fails
every allocation of a call in turn: the call must return SPMV_ERR_OOM, and the device
memory the library holds (spmv_device_memory) must be back where it was before the call.
Once k passes the call's last allocation the call succeeds, and its result is checked
against the oracle.  A failed allocation is never used: every call checks it before it
launches anything that would touch it, so the injected failure never reaches the device.
"""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_parity, to_device, torch_cuda
from workloads import integer_x, laplacian_2d, make_workload

pytestmark = pytest.mark.gpu

OOM = -4  # SPMV_ERR_OOM


def _spmv():
    import sparse_matrix_vector_csr_gb300 as spmv

    return spmv


def _fail_each(monkeypatch, call, limit=400):
    """Run call() with its 1st, 2nd, ... allocation failing until it succeeds; return
    (its result, how many allocations it made)."""
    spmv = _spmv()
    torch = torch_cuda()
    torch.cuda.synchronize()
    base = spmv.spmv_device_memory()
    for k in range(1, limit):
        monkeypatch.setenv("SPMV_FAIL_ALLOC", str(k))
        try:
            out = call()
        except spmv.SpmvError as e:
            assert e.status == OOM, (k, e)
            torch.cuda.synchronize()
            assert spmv.spmv_device_memory() == base, f"allocation {k} failed and left memory held"
            continue
        monkeypatch.delenv("SPMV_FAIL_ALLOC")
        return out, k - 1
    raise AssertionError(f"the call still failed with its {limit}-th allocation failing")


@pytest.mark.parametrize("fmt", ["auto", "sell", "hyb", "merge", "csr_vector", "ell_r"])
def test_build_releases_everything_on_each_failed_allocation(fmt, monkeypatch):
    spmv = _spmv()
    torch = torch_cuda()
    csr, _ = make_workload("powerlaw_small")
    rng = np.random.default_rng(5)
    csr = type(csr)(csr.n, csr.row_ptr, csr.col_idx, rng.integers(-8, 9, csr.nnz).astype(np.float64))
    rp, ci, vv = to_device(csr)
    torch.cuda.synchronize()
    base = spmv.spmv_device_memory()
    A, allocations = _fail_each(monkeypatch, lambda: spmv.SpmvMatrix.from_csr(rp, ci, vv, format=fmt))
    assert allocations >= 3, allocations
    assert spmv.spmv_device_memory()[0] >= base[0] + 1
    x_np = integer_x(csr.n)
    x = torch.from_numpy(x_np).cuda()
    y = torch.full_like(x, float("nan"))
    A.apply(x, y)
    torch.cuda.synchronize()
    assert_parity(y.cpu().numpy(), oracle.spmv(csr, x_np), np.float64, exact=True, label=fmt)
    A.close()
    torch.cuda.synchronize()
    assert spmv.spmv_device_memory() == base


def test_permuted_build_releases_everything(monkeypatch):
    """The RCM ordering allocates its own stream-ordered scratch before the build."""
    spmv = _spmv()
    torch = torch_cuda()
    csr = laplacian_2d(60, 50)
    rp, ci, vv = to_device(csr)
    torch.cuda.synchronize()
    base = spmv.spmv_device_memory()
    A, allocations = _fail_each(monkeypatch, lambda: spmv.SpmvMatrix.from_csr(rp, ci, vv, ordering="rcm"))
    assert allocations >= 10, allocations
    x_np = integer_x(csr.n)
    x = torch.from_numpy(x_np).cuda()
    y = A.from_basis(A.apply(A.to_basis(x)))
    torch.cuda.synchronize()
    assert_parity(y.cpu().numpy(), oracle.spmv(csr, x_np), np.float64, exact=True, label="rcm")
    A.close()
    torch.cuda.synchronize()
    assert spmv.spmv_device_memory() == base


def test_first_apply_on_a_stream_fails_cleanly(monkeypatch):
    """The first apply on a new stream allocates that stream's scratch set (row-split
    counters and partials here); when that fails the apply returns SPMV_ERR_OOM having
    launched nothing, and the next apply on the stream works."""
    spmv = _spmv()
    torch = torch_cuda()
    csr, _ = make_workload("powerlaw_small")
    rng = np.random.default_rng(6)
    csr = type(csr)(csr.n, csr.row_ptr, csr.col_idx, rng.integers(-8, 9, csr.nnz).astype(np.float64))
    rp, ci, vv = to_device(csr)
    A = spmv.SpmvMatrix.from_csr(rp, ci, vv)
    assert A.describe()["n_long_rows"] > 0
    x_np = integer_x(csr.n)
    x = torch.from_numpy(x_np).cuda()
    y = torch.full_like(x, float("nan"))
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    monkeypatch.setenv("SPMV_FAIL_ALLOC", "1")
    with pytest.raises(spmv.SpmvError) as e:
        A.apply(x, y, stream=s)
    assert e.value.status == OOM
    monkeypatch.delenv("SPMV_FAIL_ALLOC")
    torch.cuda.synchronize()
    assert torch.isnan(y).all()  # nothing ran
    A.apply(x, y, stream=s)
    s.synchronize()
    assert_parity(y.cpu().numpy(), oracle.spmv(csr, x_np), np.float64, exact=True, label="after the failure")
    A.close()


def test_solver_workspace_failure(monkeypatch):
    """CG's workspace is one stream-ordered allocation: its failure leaves nothing held."""
    spmv = _spmv()
    torch = torch_cuda()
    csr = laplacian_2d(40, 30)
    rp, ci, vv = to_device(csr)
    A = spmv.SpmvMatrix.from_csr(rp, ci, vv)
    b = torch.ones(csr.n, dtype=torch.float64, device="cuda")
    torch.cuda.synchronize()
    base = spmv.spmv_device_memory()
    monkeypatch.setenv("SPMV_FAIL_ALLOC", "1")
    with pytest.raises(spmv.SpmvError) as e:
        A.cg(b, rtol=1e-10, max_iter=500)
    assert e.value.status == OOM
    monkeypatch.delenv("SPMV_FAIL_ALLOC")
    torch.cuda.synchronize()
    assert spmv.spmv_device_memory() == base
    x, it, res = A.cg(b, rtol=1e-10, max_iter=500)
    torch.cuda.synchronize()
    assert res <= 1e-10 and it > 0
    assert spmv.spmv_device_memory() == base  # the workspace went back with the call
    A.close()


def test_plan_log(monkeypatch, capfd):
    """SPMV_LOG=1: every successful build writes its plan to stderr as one JSON line."""
    import json

    spmv = _spmv()
    csr = laplacian_2d(30, 20)
    rp, ci, vv = to_device(csr)
    monkeypatch.setenv("SPMV_LOG", "1")
    A = spmv.SpmvMatrix.from_csr(rp, ci, vv, format="sell")
    err = capfd.readouterr().err
    lines = [ln for ln in err.splitlines() if ln.startswith("spmv: built ")]
    assert len(lines) == 1, err
    plan = json.loads(lines[0][len("spmv: built "):])
    assert plan == A.describe()
    monkeypatch.setenv("SPMV_LOG", "0")
    B = spmv.SpmvMatrix.from_csr(rp, ci, vv)
    assert "spmv: built" not in capfd.readouterr().err
    A.close()
    B.close()
