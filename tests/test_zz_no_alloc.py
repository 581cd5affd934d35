"""The allocation-free entry point against the handle-based one.

spmv_csr_apply_noalloc serves callers that may not allocate device memory (for
example a program whose device memory all belongs to its own pool allocator, or a
time-critical loop that cannot take cudaMalloc's implicit synchronisation).  It
keeps its scratch in a fixed array of the library, so it is checked here on two
calls in a row (the second must not depend on what the first left there) against
spmv_apply of a handle, within the per-row tolerance of the other parity tests.
This file is collected last so a failure here cannot hide any other test.
"""
import numpy as np
import pytest

import oracle
from tests.gpu_util import build, to_device, torch_cuda
from workloads import make_workload, uniform_x

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,dtype", [("powerlaw_small", np.float64), ("hmep_small", np.float64),
                                        ("powerlaw_small", np.float32), ("lap3d_small", np.float32)])
def test_noalloc_matches_handle_on_two_calls(name, dtype):
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    csr, x0 = make_workload(name, dtype=dtype)
    rp, ci, vv = to_device(csr)
    code = 0 if dtype == np.float64 else 1
    tau = oracle.TAU[np.dtype(dtype)]
    with build(csr, "csr_vector") as A:
        for call, x_np in enumerate((x0, uniform_x(csr.n, seed=77, dtype=dtype))):
            x = torch.from_numpy(x_np).cuda()
            y_ref = A.apply(x)
            y = torch.full_like(x, float("nan"))
            spmv.spmv_csr_apply_noalloc(csr.n, csr.nnz, rp, ci, vv, code, x, y)
            torch.cuda.synchronize()
            got, want = y.cpu().numpy().astype(np.float64), y_ref.cpu().numpy().astype(np.float64)
            scale = oracle.spmv(csr, x_np)["scale"]
            # both results lie within tau * scale of the exact value
            bad = np.nonzero(~(np.abs(got - want) <= 2 * tau * scale))[0]
            assert bad.size == 0, f"call {call}: row {bad[0]} differs: {got[bad[0]]} vs {want[bad[0]]}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    tiny = torch.zeros(4, dtype=torch.int32, device="cuda")
    v = torch.zeros(4, dtype=torch.float64, device="cuda")
    with pytest.raises(spmv.SpmvError) as ei:
        spmv.spmv_csr_apply_noalloc(100_000_000, 40_000_000, tiny, tiny, v, 0, v, v)
    assert ei.value.status == -5 and "allocation-free limit" in str(ei.value)
