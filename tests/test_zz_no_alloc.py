"""The allocation-free entry point against the oracle.

spmv_csr_apply_noalloc serves callers that may not allocate device memory: a
program whose device memory all belongs to its own pool allocator, or a
time-critical loop that cannot take the implicit device synchronisation of
cudaMalloc / cudaFree.  It keeps its only scratch (the merge-path carries) in a
fixed array of the library, which every call shares and which keeps what the last
call left there.  So every case runs two calls in a row on different inputs, and
each result is compared with the oracle within the same per-row tolerance as the
other parity tests (bit for bit on integer-valued inputs); the second call must not
depend on what the first left in the scratch.  The handle-based apply is run beside
it for a cross-check.  This file is collected last, so a failure here cannot hide
any other test.
"""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_parity, build, to_device, torch_cuda
from workloads import CSR, integer_x, make_workload, uniform_x

pytestmark = pytest.mark.gpu


def _noalloc(csr, x_np, dtype):
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    rp, ci, vv = to_device(csr)
    x = torch.from_numpy(np.ascontiguousarray(x_np)).cuda()
    y = torch.full_like(x, float("nan"))  # every row must be written
    spmv.spmv_csr_apply_noalloc(csr.n, csr.nnz, rp, ci, vv, 0 if dtype == np.float64 else 1, x, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("name,dtype", [("powerlaw_small", np.float64), ("hmep_small", np.float64),
                                        ("powerlaw_small", np.float32), ("lap3d_small", np.float32)])
def test_noalloc_matches_oracle_on_two_calls(name, dtype):
    torch = torch_cuda()
    csr, x0 = make_workload(name, dtype=dtype)
    with build(csr, "csr_vector") as A:
        for call, x_np in enumerate((x0, uniform_x(csr.n, seed=77, dtype=dtype))):
            y = _noalloc(csr, x_np, dtype)
            assert_parity(y, oracle.spmv(csr, x_np), dtype, label=f"{name} call {call}")
            # cross-check: the handle's apply lies within the same bound of the oracle
            y_ref = A.apply(torch.from_numpy(x_np).cuda()).cpu().numpy()
            assert_parity(y_ref, oracle.spmv(csr, x_np), dtype, label=f"{name} handle call {call}")


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_noalloc_integer_inputs_bit_exact(dtype):
    """Integer-valued A and x: every order of summation gives the same bits."""
    csr, _ = make_workload("powerlaw_small", dtype=dtype)
    rng = np.random.default_rng(11)
    csr = CSR(csr.n, csr.row_ptr, csr.col_idx, rng.integers(-8, 9, csr.nnz).astype(dtype))
    for seed in (102, 103):
        x = integer_x(csr.n, seed=seed, dtype=dtype)
        assert_parity(_noalloc(csr, x, dtype), oracle.spmv(csr, x), dtype, exact=True, label=f"seed {seed}")


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_noalloc_single_row_of_a_million(dtype):
    """One row of 10^6 entries spans about 490 merge-path shares: the carry fix-up walks
    a run of carries longer than a warp, on two calls in a row."""
    n = 1_000_000
    row_ptr = np.full(n + 1, n, dtype=np.int32)
    row_ptr[0] = 0
    rng = np.random.default_rng(5)
    rows = np.arange(0, n, 997)
    for integer in (True, False):
        vals = (rng.integers(-8, 9, n) if integer else rng.standard_normal(n)).astype(dtype)
        csr = CSR(n, row_ptr, np.arange(n, dtype=np.int32), vals)
        x = integer_x(n, dtype=dtype) if integer else uniform_x(n, dtype=dtype)
        y = _noalloc(csr, x, dtype)
        assert_parity(y[rows], oracle.spmv(csr, x, rows=rows), dtype, exact=integer, label=f"integer={integer}")
        assert np.all(y[1:] == 0) and not np.signbit(y[1:]).any()  # empty rows give +0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    tiny = torch.zeros(4, dtype=torch.int32, device="cuda")
    v = torch.zeros(4, dtype=torch.float64, device="cuda")
    with pytest.raises(spmv.SpmvError) as ei:
        spmv.spmv_csr_apply_noalloc(100_000_000, 40_000_000, tiny, tiny, v, 0, v, v)
    assert ei.value.status == -5 and "allocation-free limit" in str(ei.value)


def test_noalloc_refuses_overlapping_output():
    """y must not overlap x (an in-place call) nor the matrix arrays: other shares of the
    work are still reading them while y is written."""
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    csr, x_np = make_workload("lap3d_small")
    rp, ci, vv = to_device(csr)
    x = torch.from_numpy(x_np).cuda()
    for y in (x, x[3:], vv):
        with pytest.raises(spmv.SpmvError) as ei:
            spmv.spmv_csr_apply_noalloc(csr.n, csr.nnz, rp, ci, vv, 0, x, y)
        assert ei.value.status == -1 and "overlap" in str(ei.value)
    # a view that ends right where x starts does not overlap it
    buf = torch.empty(2 * csr.n, dtype=torch.float64, device="cuda")
    buf[csr.n:] = x
    spmv.spmv_csr_apply_noalloc(csr.n, csr.nnz, rp, ci, vv, 0, buf[csr.n:], buf[:csr.n])
    torch.cuda.synchronize()
    assert_parity(buf[:csr.n].cpu().numpy(), oracle.spmv(csr, x_np), np.float64, label="adjacent buffers")
