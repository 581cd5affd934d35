"""The permuted basis (spmv_build_permuted, spmv_get_permutation, spmv_permute_vector)
against the ordering oracle: orderings and B = P A P^T bit-exact (integer and index
work), products in the permuted basis within the per-row tolerance, a CG solve in the
permuted basis, and, at full size, properties of the reverse Cuthill-McKee order that
hold at any size."""
import numpy as np
import pytest

import oracle
from oracle import ordering as ordr
from oracle.cg import cg as oracle_cg
from tests.gpu_util import assert_parity, case_id, to_device, torch_cuda
from workloads import CSR, make_workload, random_csr, uniform_x

pytestmark = pytest.mark.gpu

_cache = {}


def workload(name):
    if name not in _cache:
        if name == "components":
            csr = random_csr(3000, density=0.0004, seed=21, duplicates=True, unsorted=True, empty_row_fraction=0.05)
            _cache[name] = (csr, uniform_x(csr.n, seed=5))
        else:
            _cache[name] = make_workload(name)
    return _cache[name]


def oracle_order(csr, kind):
    return ordr.reverse_cuthill_mckee(csr) if kind == "rcm" else ordr.row_length_order(csr)


def build(csr, fmt="auto", ordering="rcm", **params):
    import sparse_matrix_vector_csr_gb300 as spmv

    rp, ci, vv = to_device(csr)
    return spmv.SpmvMatrix.from_csr(rp, ci, vv, format=fmt, ordering=ordering, **params)


ORDER_CASES = [("lap2d_small", "rcm"), ("lap3d_relabelled_small", "rcm"), ("powerlaw_small", "rcm"),
               ("band_small", "rcm"), ("components", "rcm"), ("hmep_small", "row_length"),
               ("powerlaw_small", "row_length"), ("lap3d_relabelled_small", "row_length")]


@pytest.mark.parametrize("name,kind", ORDER_CASES)
def test_permutation_and_permuted_matrix(name, kind):
    csr, _ = workload(name)
    expect = oracle_order(csr, kind)
    B_ref = ordr.symmetric_permute(csr, expect)
    with build(csr, ordering=kind) as A:
        d = A.describe()
        assert d["ordering"] == kind and d["permuted_basis"]
        assert np.array_equal(A.permutation().cpu().numpy(), expect)
        rp, ci, vv = (t.cpu().numpy() for t in A.to_csr())
        assert np.array_equal(rp, B_ref.row_ptr) and np.array_equal(ci, B_ref.col_idx)
        assert np.array_equal(vv.view(np.uint8), B_ref.vals.view(np.uint8))


FORMATS = [("auto", {}), ("csr_vector", {}), ("hyb", {}), ("merge", {}), ("sell", {"row_threads": 4}),
           ("sell", {"C": 64, "sigma": 1 << 30})]


@pytest.mark.parametrize("fmt,params", FORMATS, ids=[case_id(c) for c in FORMATS])
@pytest.mark.parametrize("name", ["lap3d_relabelled_small", "powerlaw_small", "components"])
def test_products_in_the_permuted_basis(name, fmt, params):
    torch = torch_cuda()
    csr, x = workload(name)
    perm = ordr.reverse_cuthill_mckee(csr)
    B = ordr.symmetric_permute(csr, perm)
    with build(csr, fmt, "rcm", **params) as A:
        xd = torch.from_numpy(x).cuda()
        xp = A.to_basis(xd)
        assert np.array_equal(xp.cpu().numpy(), x[perm])
        yp = A.apply(xp)
        torch.cuda.synchronize()
        assert_parity(yp.cpu().numpy(), oracle.spmv(B, x[perm]), np.float64, label=f"{name}/{fmt}")
        y = A.from_basis(yp)
        torch.cuda.synchronize()
        assert_parity(y.cpu().numpy(), oracle.spmv(csr, x), np.float64, label=f"{name}/{fmt} original basis")
        back = A.from_basis(xp)
        assert np.array_equal(back.cpu().numpy().view(np.uint64), x.view(np.uint64))


def test_user_ordering_and_errors():
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    csr, x = workload("lap2d_small")
    perm = np.random.default_rng(3).permutation(csr.n).astype(np.int32)
    with build(csr, ordering=torch.from_numpy(perm).cuda()) as A:
        assert np.array_equal(A.permutation().cpu().numpy(), perm)
        assert A.describe()["ordering"] == "user"
        y = A.from_basis(A.apply(A.to_basis(torch.from_numpy(x).cuda())))
        torch.cuda.synchronize()
        assert_parity(y.cpu().numpy(), oracle.spmv(csr, x), np.float64)
    bad = perm.copy()
    bad[5] = bad[6]
    with pytest.raises(spmv.SpmvError) as ei:
        build(csr, ordering=torch.from_numpy(bad).cuda())
    assert ei.value.status == -1
    bad[5] = csr.n
    with pytest.raises(spmv.SpmvError):
        build(csr, ordering=torch.from_numpy(bad).cuda())
    broken = CSR(csr.n, csr.row_ptr, np.where(np.arange(csr.nnz) == 7, csr.n + 3, csr.col_idx).astype(np.int32),
                 csr.vals)
    with pytest.raises(spmv.SpmvError) as ei:
        build(broken, ordering="rcm")
    assert ei.value.status == -2


def test_natural_and_plain_handles_are_identity():
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    csr, x = workload("lap2d_small")
    with build(csr, ordering="natural") as A:
        assert np.array_equal(A.permutation().cpu().numpy(), np.arange(csr.n))
    rp, ci, vv = to_device(csr)
    with spmv.SpmvMatrix.from_csr(rp, ci, vv) as A:
        assert not A.describe()["permuted_basis"]
        assert np.array_equal(A.permutation().cpu().numpy(), np.arange(csr.n))
        xd = torch.from_numpy(x).cuda()
        assert torch.equal(A.to_basis(xd), xd)


def test_diagonal_and_empty_matrices():
    torch = torch_cuda()
    n = 1000
    diag = CSR(n, np.arange(n + 1, dtype=np.int32), np.arange(n, dtype=np.int32), np.arange(1.0, n + 1))
    with build(diag, ordering="rcm") as A:
        assert np.array_equal(A.permutation().cpu().numpy(), np.arange(n)[::-1])
    empty = CSR(n, np.zeros(n + 1, np.int32), np.zeros(0, np.int32), np.zeros(0))
    with build(empty, ordering="rcm") as A:
        assert np.array_equal(A.permutation().cpu().numpy(), ordr.reverse_cuthill_mckee(empty))
        y = A.apply(torch.ones(n, dtype=torch.float64, device="cuda"))
        assert not y.any()


def test_cg_in_the_permuted_basis():
    torch = torch_cuda()
    csr, _ = workload("lap3d_relabelled_small")
    b = uniform_x(csr.n, seed=41)
    with build(csr, ordering="rcm") as A:
        bp = A.to_basis(torch.from_numpy(b).cuda())
        xp, it, res = A.cg(bp, rtol=1e-8, max_iter=2000)
        x = A.from_basis(xp).cpu().numpy()
    ref = oracle_cg(csr, b, rtol=1e-8, max_iter=2000)
    r = b - oracle.spmv(csr, x)["y_hi"]
    assert np.linalg.norm(r) / np.linalg.norm(b) <= 1.01e-8
    assert abs(it - ref["iterations"]) <= 2


def _max_plane(nx, ny, nz):
    i, j, k = np.meshgrid(np.arange(nx), np.arange(ny), np.arange(nz), indexing="ij")
    return int(np.bincount((i + j + k).ravel()).max())


def test_full_size_rcm_on_the_relabelled_128_cube():
    """At 128^3: a permutation; every edge joins adjacent breadth-first levels (planes
    i + j + k = s from a corner), so the bandwidth of B is below twice the largest plane;
    sampled rows of the product in the permuted basis against the oracle."""
    torch = torch_cuda()
    csr, x = make_workload("lap3d_128_relabelled")
    with build(csr, ordering="rcm") as A:
        perm = A.permutation().cpu().numpy()
        assert np.array_equal(np.sort(perm), np.arange(csr.n))
        rp, ci, vv = A.to_csr()
        rows = torch.repeat_interleave(torch.arange(csr.n, device="cuda"), rp[1:] - rp[:-1])
        bw = int((rows - ci.long()).abs().max())
        assert bw < 2 * _max_plane(128, 128, 128)
        xp = A.to_basis(torch.from_numpy(x).cuda())
        yp = A.apply(xp).cpu().numpy()
        B = CSR(csr.n, rp.cpu().numpy(), ci.cpu().numpy(), vv.cpu().numpy())
        sample = np.random.default_rng(8).choice(csr.n, 20000, replace=False)
        ref = oracle.spmv(B, x[perm], rows=sample)
        assert_parity(yp[sample], ref, np.float64, label="lap3d_128_relabelled rcm")
