"""Host-buffer entry points against the oracle: the staging-copy path (spmv_apply_host)
and the mapped path (spmv_apply_mapped, the kernels reading and writing page-locked host
memory directly), on several formats; host memory that is not page-locked is refused."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_parity, build, case_id, torch_cuda
from workloads import make_workload

pytestmark = pytest.mark.gpu

CASES = [("auto", {}), ("merge", {}), ("csr_vector", {}), ("hyb", {"spill_csr": 0}), ("sell", {"row_threads": 4})]


@pytest.mark.parametrize("fmt,params", CASES, ids=[case_id(c) for c in CASES])
@pytest.mark.parametrize("name", ["powerlaw_small", "hmep_small", "uniform16_small"])
def test_mapped_and_copy_paths(name, fmt, params):
    torch = torch_cuda()
    csr, x = make_workload(name)
    ref = oracle.spmv(csr, x)
    with build(csr, fmt, **params) as A:
        xt = torch.from_numpy(x).pin_memory()
        yt = torch.full_like(xt, float("nan")).pin_memory()
        A.apply_mapped(xt, yt)
        assert_parity(yt.numpy(), ref, csr.dtype, label=f"mapped {name}/{fmt}")
        yh = np.full_like(x, np.nan)  # pageable: staged and copied back
        A.apply_host(xt.numpy(), yh)
        assert_parity(yh, ref, csr.dtype, label=f"copy {name}/{fmt}")
        assert np.array_equal(yh.view(np.uint8), yt.numpy().view(np.uint8))  # same kernels, same bits
        yp = torch.full_like(xt, float("nan")).pin_memory()  # page-locked: stored directly when the plan allows
        A.apply_host(xt.numpy(), yp.numpy())
        assert np.array_equal(yp.numpy().view(np.uint8), yh.view(np.uint8))


def test_mapped_refuses_pageable_and_device_memory():
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    csr, x = make_workload("lap2d_small")
    with build(csr) as A:
        y = np.empty_like(x)
        with pytest.raises(spmv.SpmvError) as ei:
            spmv.spmv_apply_mapped(A._h, x, y)  # ordinary numpy memory
        assert ei.value.status == -1
        xd = torch.from_numpy(x).cuda()
        with pytest.raises(spmv.SpmvError):
            spmv.spmv_apply_mapped(A._h, xd, torch.empty_like(xd))
