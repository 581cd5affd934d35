"""Randomised plans: seeded random matrices (sizes across several tiles with ragged
tails, empty and full rows, duplicates, unsorted rows, a few long rows) built with
random formats and parameters (threads per row and their mode, vector loads, the x
cache policy, row blocks of the pipelined host path), in both value types, against the
oracle: the product within the per-row tolerance, the round trip to CSR array for
array, y = alpha A x + beta y, and the host-array apply bit for bit equal to the device
apply.  Every case is seeded, so a failure names a reproducible configuration."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_parity, assert_roundtrip, build, torch_cuda
from workloads import CSR, random_csr, uniform_x

pytestmark = pytest.mark.gpu


def random_plan(rng):
    fmt = rng.choice(["auto", "csr_vector", "ell_r", "sell", "hyb", "merge"])
    p = {}
    if fmt in ("sell",):
        p["C"] = int(rng.choice([32, 64, 128]))
        p["sigma"] = int(rng.choice([1, 2, 32, 256, 1000, 1 << 30]))
    if fmt in ("sell", "ell_r", "hyb") and rng.random() < 0.6:
        g = int(rng.choice([1, 2, 4, 8, 16, 32]))
        p["row_threads"] = g
        p["row_group_mode"] = int(rng.choice([0, 1, 2] if g <= 8 else [0, 1]))
    elif fmt in ("sell", "ell_r", "hyb") and rng.random() < 0.6:
        p["vector_loads"] = 1
    if fmt in ("sell", "ell_r", "hyb") and rng.random() < 0.3:
        p["x_policy"] = int(rng.integers(0, 2))
    if fmt in ("sell", "ell_r") and rng.random() < 0.7:
        p["host_blocks"] = int(rng.choice([2, 3, 5, 16]))
    if fmt in ("sell", "ell_r", "csr_vector") and rng.random() < 0.5:
        p["long_row_threshold"] = int(rng.choice([0, 4, 16, 100]))
    if fmt == "csr_vector" and rng.random() < 0.4:
        p["subwarp"] = int(rng.choice([2, 4, 8, 16, 32]))
    if fmt == "hyb" and rng.random() < 0.6:
        p["K"] = int(rng.integers(0, 12))
        p["spill_csr"] = int(rng.integers(0, 2))
    return str(fmt), p


def random_matrix(rng, seed):
    n = int(rng.choice([1, 7, 33, 257, 1000, 3001, 9000]))
    density = float(rng.choice([0.0, 0.001, 0.01, 0.05, 0.3])) if n > 1 else 1.0
    csr = random_csr(n, density, seed=seed, duplicates=bool(rng.random() < 0.3), unsorted=bool(rng.random() < 0.3),
                     empty_row_fraction=float(rng.choice([0.0, 0.2])), full_rows=int(rng.integers(0, 3)) if n > 1 else 0)
    if n > 100 and rng.random() < 0.5:
        # a few long rows next to short ones
        lens = np.diff(csr.row_ptr.astype(np.int64))
        long_rows = rng.choice(n, size=3, replace=False)
        lens[long_rows] = rng.integers(n // 4, n, size=3)
        row_ptr = np.zeros(n + 1, np.int64)
        np.cumsum(lens, out=row_ptr[1:])
        cols = rng.integers(0, n, size=int(row_ptr[-1])).astype(np.int32)
        vals = rng.standard_normal(cols.size)
        csr = CSR(n, row_ptr.astype(np.int32), cols, vals)
    return csr


@pytest.mark.parametrize("seed", range(160))
def test_random_plan(seed):
    torch = torch_cuda()
    rng = np.random.default_rng(1000 + seed)
    csr = random_matrix(rng, seed)
    dtype = np.float32 if rng.random() < 0.4 else np.float64
    csr = csr.astype(dtype)
    fmt, params = random_plan(rng)
    x = uniform_x(csr.n, seed=seed, dtype=dtype)
    label = f"seed {seed}: n={csr.n} nnz={csr.nnz} {np.dtype(dtype).name} {fmt} {params}"
    with build(csr, fmt, **params) as A:
        xd = torch.from_numpy(x).cuda()
        y = torch.full_like(xd, float("nan"))
        A.apply(xd, y)
        torch.cuda.synchronize()
        assert_parity(y.cpu().numpy(), oracle.spmv(csr, x), dtype, label=label)
        assert_roundtrip(A, csr, label=label)
        alpha, beta = float(rng.choice([-1.0, 0.5, 2.0])), float(rng.choice([0.0, 1.0, -0.25]))
        y0 = uniform_x(csr.n, seed=seed + 7, dtype=dtype)
        yd = torch.from_numpy(y0.copy()).cuda()
        A.apply(xd, yd, alpha=alpha, beta=beta)
        torch.cuda.synchronize()
        assert_parity(yd.cpu().numpy(), oracle.spmv_scaled(csr, x, alpha, beta, y0), dtype, label=label + " scaled")
        xh = torch.from_numpy(x).pin_memory()
        yh = torch.full_like(xh, float("nan")).pin_memory()
        A.apply_host(xh.numpy(), yh.numpy())
        assert np.array_equal(yh.numpy().view(np.uint8), y.cpu().numpy().view(np.uint8)), label + " host"
