"""y = alpha A x + beta y (spmv_apply_ex) and Y = alpha A X + beta Y (spmv_apply_multi)
against the oracle, on every format, both value types, fused and column-by-column paths."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import FORMAT_CASES, assert_parity, build, case_id, torch_cuda
from workloads import integer_x, laplacian_2d, make_workload, uniform_x

pytestmark = pytest.mark.gpu

SCALES = [(-1.0, 1.0), (2.5, -0.5), (0.0, 3.0), (-3.0, 0.0)]
MULTI_FORMATS = [("auto", {}), ("sell", {"C": 64, "sigma": 256}), ("sell", {"C": 32, "sigma": 1 << 30}),
                 ("ell_r", {}), ("hyb", {}), ("merge", {}), ("csr_vector", {}), ("sell", {"row_threads": 4})]

_cache = {}


def small(name, dtype=None):
    key = (name, dtype)
    if key not in _cache:
        _cache[key] = make_workload(name, dtype=dtype)
    return _cache[key]


def flat(ref):
    return {k: np.ascontiguousarray(v).reshape(-1) for k, v in ref.items()}


@pytest.mark.parametrize("case", FORMAT_CASES, ids=case_id)
@pytest.mark.parametrize("name", ["powerlaw_small", "hmep_small"])
def test_scaled_every_format(name, case):
    torch = torch_cuda()
    fmt, params = case
    csr, x = small(name)
    y_old = uniform_x(csr.n, seed=31)
    with build(csr, fmt, **params) as A:
        xd = torch.from_numpy(x).cuda()
        for alpha, beta in SCALES:
            y = torch.from_numpy(y_old).cuda() if beta != 0 else torch.full_like(xd, float("nan"))
            A.apply(xd, y, alpha=alpha, beta=beta)
            torch.cuda.synchronize()
            ref = oracle.spmv_scaled(csr, x, alpha, beta, y_old)
            assert_parity(y.cpu().numpy(), ref, np.float64, label=f"{name}/{case_id(case)} a={alpha} b={beta}")


@pytest.mark.parametrize("case", FORMAT_CASES, ids=case_id)
def test_scaled_integer_exact(case):
    torch = torch_cuda()
    fmt, params = case
    csr = laplacian_2d(256, 256)
    x = integer_x(csr.n)
    b = integer_x(csr.n, seed=77)
    with build(csr, fmt, **params) as A:
        r = torch.from_numpy(b).cuda()
        A.apply(torch.from_numpy(x).cuda(), r, alpha=-1.0, beta=1.0)  # residual b - A x
        torch.cuda.synchronize()
        ref = oracle.spmv_scaled(csr, x, -1.0, 1.0, b)
        assert_parity(r.cpu().numpy(), ref, np.float64, exact=True, label=case_id((fmt, params)))


@pytest.mark.parametrize("fmt,params", MULTI_FORMATS, ids=[case_id(c) for c in MULTI_FORMATS])
@pytest.mark.parametrize("k", [1, 2, 3, 4, 5, 8, 13, 16])
@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_multi_vector(fmt, params, k, dtype):
    torch = torch_cuda()
    csr, _ = small("powerlaw_small", dtype)
    rng = np.random.default_rng(k)
    X = (rng.random((csr.n, k)) * 2 - 1).astype(dtype)
    Y0 = (rng.random((csr.n, k)) * 2 - 1).astype(dtype)
    alpha, beta = (1.0, 0.0) if k % 2 else (-0.75, 2.0)
    with build(csr, fmt, **params) as A:
        Xd = torch.from_numpy(X).cuda()
        Yd = torch.from_numpy(Y0).cuda() if beta != 0 else torch.full_like(Xd, float("nan"))
        A.apply_multi(Xd, Yd, alpha=alpha, beta=beta)
        torch.cuda.synchronize()
        ref = oracle.spmm(csr, X, alpha, beta, Y0)
        assert_parity(Yd.cpu().numpy().reshape(-1), flat(ref), dtype, label=f"{fmt} {params} k={k}")


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_multi_vector_strided_and_misaligned(dtype):
    """X and Y as column slices of wider blocks: odd leading dimensions and an X base that is
    not 16-byte aligned take the column-by-column path; results must not change."""
    torch = torch_cuda()
    csr, _ = small("hmep_small", dtype)
    rng = np.random.default_rng(5)
    big = (rng.random((csr.n, 11)) * 2 - 1).astype(dtype)
    k = 6
    with build(csr, "auto") as A:
        Bd = torch.from_numpy(big).cuda()
        for start in (0, 1, 3):
            Xd = Bd[:, start:start + k]                    # ldx = 11, base offset `start` values
            Yd = torch.full((csr.n, 13), float("nan"), dtype=Xd.dtype, device="cuda")[:, 2:2 + k]
            A.apply_multi(Xd, Yd)
            torch.cuda.synchronize()
            ref = oracle.spmm(csr, big[:, start:start + k])
            assert_parity(Yd.cpu().numpy().reshape(-1), flat(ref), dtype, label=f"start={start}")


@pytest.mark.parametrize("fmt,params", MULTI_FORMATS, ids=[case_id(c) for c in MULTI_FORMATS])
def test_multi_vector_integer_exact(fmt, params):
    torch = torch_cuda()
    csr, _ = small("powerlaw_small")
    csr = type(csr)(csr.n, csr.row_ptr, csr.col_idx,
                    np.random.default_rng(3).integers(-8, 9, csr.nnz).astype(np.float64))
    X = np.random.default_rng(4).integers(-8, 9, (csr.n, 8)).astype(np.float64)
    with build(csr, fmt, **params) as A:
        Yd = A.apply_multi(torch.from_numpy(X).cuda())
        torch.cuda.synchronize()
        ref = oracle.spmm(csr, X)
        assert_parity(Yd.cpu().numpy().reshape(-1), flat(ref), np.float64, exact=True, label=fmt)


def test_multi_vector_in_a_cuda_graph():
    torch = torch_cuda()
    csr, _ = small("powerlaw_small")
    X = uniform_x(csr.n * 4, seed=9).reshape(csr.n, 4)
    with build(csr, "auto") as A:
        Xd = torch.from_numpy(X).cuda()
        Yd = torch.empty_like(Xd)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            A.apply_multi(Xd, Yd)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            A.apply_multi(Xd, Yd)
            A.apply_multi(Xd, Yd)
        Yd.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_parity(Yd.cpu().numpy().reshape(-1), flat(oracle.spmm(csr, X)), np.float64, label="graph")
