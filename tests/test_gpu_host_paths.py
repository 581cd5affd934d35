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


# --------------------------------------------------------------------------- #
# pipelined spmv_apply_host: pieces of x in, blocks of rows multiplied as their columns
# arrive, rows of y back on a second copy stream
# --------------------------------------------------------------------------- #
PIPE_CASES = [("sell", {"C": 32, "sigma": 1}), ("sell", {"C": 64, "sigma": 1}), ("sell", {"C": 32, "sigma": 64}),
              ("sell", {"C": 64, "sigma": 96}), ("ell_r", {}), ("auto", {})]


def host_apply(A, x, pinned_y=True):
    torch = torch_cuda()
    xt = torch.from_numpy(x).pin_memory()
    y = torch.full_like(xt, float("nan")).pin_memory().numpy() if pinned_y else np.full_like(x, np.nan)
    A.apply_host(xt.numpy(), y)
    return y


def device_apply(A, x):
    torch = torch_cuda()
    y = A.apply(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("blocks", [2, 3, 7, 16])
@pytest.mark.parametrize("fmt,params", PIPE_CASES, ids=[case_id(c) for c in PIPE_CASES])
@pytest.mark.parametrize("name", ["lap3d_small", "lap3d_relabelled_small", "hmep_small"])
def test_pipelined_apply_host(name, fmt, params, blocks):
    """Every block layout (slice heights, sort windows, ELLPACK-R's one slice, a ragged
    last block) gives the device apply's result bit for bit, and the oracle's within the
    per-row tolerance; a second call reuses the streams and events."""
    csr, x = make_workload(name)
    with build(csr, fmt, host_blocks=blocks, **params) as A:
        y = host_apply(A, x)
        d = A.describe()
        assert d["host_blocks"] == blocks and d["host_pipeline_blocks"] >= 2, d
        assert_parity(y, oracle.spmv(csr, x), csr.dtype, label=f"pipelined {name}/{fmt}/{blocks}")
        yd = device_apply(A, x)
        assert np.array_equal(y.view(np.uint8), yd.view(np.uint8))
        x2 = x[::-1].copy()
        y2 = host_apply(A, x2)
        assert np.array_equal(y2.view(np.uint8), device_apply(A, x2).view(np.uint8))


def expected_reach(csr, block):
    """For each block of `block` rows, the piece of x (same boundaries) holding its largest column."""
    nb = -(-csr.n // block)
    out = []
    for b in range(nb):
        lo, hi = csr.row_ptr[b * block], csr.row_ptr[min(csr.n, (b + 1) * block)]
        out.append(int(csr.col_idx[lo:hi].max()) // block if hi > lo else -1)
    return out


REACH_CASES = [(name, fmt, params) for name in ("lap3d_small", "lap3d_relabelled_small", "hmep_small")
               for fmt, params in PIPE_CASES[:5]] + [("powerlaw_small", fmt, params) for fmt, params in PIPE_CASES[:4]]


@pytest.mark.parametrize("name,fmt,params", REACH_CASES, ids=[f"{n}-{case_id((f, p))}" for n, f, p in REACH_CASES])
def test_pipeline_block_reach(name, fmt, params):
    """The device's column reach of every block (which piece of x the block waits for)
    equals the largest column of the block's rows, computed here from the CSR."""
    csr, x = make_workload(name)
    with build(csr, fmt, host_blocks=6, long_row_threshold=0, **params) as A:
        host_apply(A, x)
        d = A.describe()
        assert d["host_pipeline_blocks"] >= 2, d
        block = d["host_pipeline_block_rows"]
        reach = d["host_pipeline_reach"]
        assert len(reach) == d["host_pipeline_blocks"]
        exp = expected_reach(csr, block)
        assert reach[:len(exp)] == exp and all(r == -1 for r in reach[len(exp):])


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_pipelined_reach_far_columns(dtype):
    """Rows that reach the last piece of x (a random matrix with empty rows and
    duplicates): every block waits for the whole of x, and the result is unchanged."""
    from workloads import random_csr

    csr = random_csr(9000, 0.002, seed=31, duplicates=True, unsorted=True, empty_row_fraction=0.2).astype(dtype)
    x = np.random.default_rng(32).uniform(-1, 1, csr.n).astype(dtype)
    with build(csr, "sell", C=32, sigma=1, host_blocks=5) as A:
        y = host_apply(A, x)
        assert A.describe()["host_pipeline_blocks"] == 5
        assert_parity(y, oracle.spmv(csr, x), dtype, label="pipelined random")
        assert np.array_equal(y.view(np.uint8), device_apply(A, x).view(np.uint8))


def test_unpipelined_cases():
    """host_blocks = 0 or 1, pageable y, a plan with a separate pass, or one sort window
    covering every row run unpipelined, with the same result."""
    csr, x = make_workload("lap3d_small")
    ref = oracle.spmv(csr, x)
    for fmt, params, pinned in [("sell", {"host_blocks": 0}, True), ("sell", {"host_blocks": 1}, True),
                                ("sell", {"host_blocks": 4}, False), ("merge", {"host_blocks": 4}, True),
                                ("hyb", {"host_blocks": 4, "K": 3}, True),
                                ("sell", {"host_blocks": 4, "row_threads": 4}, True),
                                ("sell", {"host_blocks": 4, "sigma": 1 << 30}, True)]:
        with build(csr, fmt, **params) as A:
            y = host_apply(A, x, pinned_y=pinned)
            assert A.describe()["host_pipeline_blocks"] == 0, (fmt, params, pinned)
            assert_parity(y, ref, csr.dtype, label=f"unpipelined {fmt} {params}")


def test_host_blocks_argument_checked():
    import sparse_matrix_vector_csr_gb300 as spmv

    csr, _ = make_workload("lap2d_small")
    with pytest.raises(spmv.SpmvError) as ei:
        build(csr, "sell", host_blocks=4096)
    assert ei.value.status == -1


def test_pipeline_at_size_and_default_off():
    """A 96^3 Laplacian (x = 7 MB) in 8 blocks, each reaching one piece of x ahead: the
    device apply's result bit for bit, sampled rows against the oracle.  Without
    host_blocks the call is unpipelined."""
    from workloads import laplacian_3d

    lap = laplacian_3d(96, 96, 96)
    x = np.random.default_rng(41).uniform(-1, 1, lap.n)
    with build(lap, "auto", host_blocks=8) as A:
        assert A.describe()["host_pipeline_blocks"] == -1  # no call yet
        y = host_apply(A, x)
        assert A.describe()["host_pipeline_blocks"] == 8
        assert np.array_equal(y.view(np.uint8), device_apply(A, x).view(np.uint8))
        sample = np.random.default_rng(42).choice(lap.n, 20000, replace=False)
        assert_parity(y[sample], oracle.spmv(lap, x, rows=sample), np.float64, label="96^3 pipelined")
    with build(lap, "auto") as A:
        y0 = host_apply(A, x)
        d = A.describe()
        assert d["host_blocks"] == 0 and d["host_pipeline_blocks"] == 0
        assert np.array_equal(y0.view(np.uint8), y.view(np.uint8))


def test_overlapping_vectors():
    """Overlapping x and y are refused by the device and mapped entry points; the host
    path computes in place (unpipelined even with host_blocks set)."""
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    csr, x = make_workload("lap3d_small")
    ref = oracle.spmv(csr, x)
    with build(csr, "sell", host_blocks=4) as A:
        xd = torch.from_numpy(x).cuda()
        for y in (xd, xd[1:]):  # the same array, and one shifted by an element
            with pytest.raises(spmv.SpmvError) as ei:
                spmv.spmv_apply(A._h, xd, y)
            assert ei.value.status == -1
        with pytest.raises(spmv.SpmvError):
            spmv.spmv_apply_ex(A._h, 2.0, xd, 1.0, xd)
        X = torch.zeros(csr.n, 4, dtype=xd.dtype, device="cuda")
        with pytest.raises(spmv.SpmvError):
            spmv.spmv_apply_multi(A._h, 2, 1.0, X, 4, 0.0, X[:, 2:], 4)
        Y = torch.zeros_like(X)
        spmv.spmv_apply_multi(A._h, 2, 1.0, X, 4, 0.0, Y, 4)  # disjoint: accepted
        xt = torch.from_numpy(x).pin_memory()
        with pytest.raises(spmv.SpmvError):
            spmv.spmv_apply_mapped(A._h, xt, xt)
        buf = xt.clone().pin_memory()
        A.apply_host(buf.numpy(), buf.numpy())  # in place
        assert A.describe()["host_pipeline_blocks"] == 0
        assert_parity(buf.numpy(), ref, csr.dtype, label="in place")
        y = host_apply(A, x)
        assert A.describe()["host_pipeline_blocks"] == 4
        assert np.array_equal(y.view(np.uint8), buf.numpy().view(np.uint8))


def test_host_arrays_checked():
    """Host arrays of the wrong length, type or layout are refused before any copy."""
    torch = torch_cuda()
    csr, x = make_workload("lap2d_small")
    with build(csr) as A:
        good = np.empty_like(x)
        for bad_x in (x[:-1], x.astype(np.float32), np.stack([x, x], axis=1)[:, 0], [0.0] * csr.n):
            with pytest.raises(ValueError):
                A.apply_host(bad_x, good)
        ro = np.empty_like(x)
        ro.flags.writeable = False
        with pytest.raises(ValueError):
            A.apply_host(x, ro)
        xt = torch.from_numpy(x).pin_memory()
        with pytest.raises(ValueError):
            A.apply_mapped(xt, torch.empty(csr.n - 1, dtype=xt.dtype).pin_memory())
        y = A.apply_host(x)
        assert_parity(y, oracle.spmv(csr, x), csr.dtype, label="checked host arrays")
