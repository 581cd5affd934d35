"""The narrow-tail path of globally sorted SELL-32 layouts, and the measurement entry points.

With every row sorted by length (sigma >= n) the last slices hold rows of at most two
entries; the apply takes them two rows a thread with slot addresses from a table of
width regions instead of the slice offsets.  Those slices mix rows of length 2, 1 and 0
(a width-2 slice may hold length-1 rows, whose second slot is padding with column 0),
and the rows longer than the threshold, which the row-split pass handles, sort to the
very end with the empty rows (length -1 in the layout).  Every case checks the oracle
within tolerance, or bit for bit on integer data, with y prefilled with NaN and x
holding +Inf / NaN at the columns only padding could reach.
"""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_parity, build, run, torch_cuda
from workloads import CSR, uniform_x

pytestmark = pytest.mark.gpu


def _tail_matrix(n, seed, dtype, integer, long_rows=6):
    """Rows of 0, 1 and 2 entries mostly, some of 3..40, and a few long rows (> 128).
    Columns from 2 on, so x[0] and x[1] are referenced by no stored entry."""
    rng = np.random.default_rng(seed)
    lens = rng.choice([0, 1, 2, 3, 7, 40], size=n, p=[0.15, 0.45, 0.25, 0.08, 0.05, 0.02])
    lens[rng.choice(n, long_rows, replace=False)] = rng.integers(300, min(9000, n - 2), long_rows)
    rows = [np.sort(rng.choice(np.arange(2, n), int(k), replace=False)) for k in lens]
    rp = np.zeros(n + 1, np.int64)
    np.cumsum(lens, out=rp[1:])
    col = np.concatenate(rows).astype(np.int32)
    vals = (rng.integers(-8, 9, col.size) if integer else rng.standard_normal(col.size)).astype(dtype)
    return CSR(n, rp.astype(np.int32), col, vals)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("integer", [True, False], ids=["integer", "real"])
@pytest.mark.parametrize("n", [4099, 70001])
def test_tail_path_matches_oracle(n, integer, dtype):
    csr = _tail_matrix(n, seed=n, dtype=dtype, integer=integer)
    rng = np.random.default_rng(3)
    x = (rng.integers(-8, 9, n) if integer else uniform_x(n, seed=5)).astype(dtype)
    x[0], x[1] = np.inf, np.nan  # columns no stored entry uses: padding must not reach them
    for fmt, params in (("auto", {}), ("sell", {"C": 32, "sigma": 1 << 30})):
        with build(csr, fmt, **params) as A:
            d = A.describe()
            assert d["permuted"] and d["tail_positions"] > 0 and d["n_long_rows"] > 0, d
            y = run(A, x)
            assert np.all(np.isfinite(y))
            assert_parity(y, oracle.spmv(csr, x), dtype, exact=integer, label=f"{fmt} n={n}")


def test_tail_path_scaled_apply():
    """y = alpha A x + beta y through the tail path's fused epilogue (beta = 0 never reads y)."""
    torch = torch_cuda()
    n = 20011
    csr = _tail_matrix(n, seed=7, dtype=np.float64, integer=True)
    x = np.random.default_rng(8).integers(-8, 9, n).astype(np.float64)
    y0 = np.random.default_rng(9).integers(-8, 9, n).astype(np.float64)
    ax = oracle.spmv(csr, x)["y_hi"]
    with build(csr, "auto") as A:
        assert A.describe()["tail_positions"] > 0
        xd = torch.from_numpy(x).cuda()
        y = torch.from_numpy(y0).cuda()
        A.apply(xd, y, alpha=-2.0, beta=0.5)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), -2.0 * ax + 0.5 * y0)
        y.fill_(float("nan"))
        A.apply(xd, y, alpha=3.0, beta=0.0)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), 3.0 * ax)


def test_tail_of_only_empty_and_unit_rows():
    """Every row has 0 or 1 entries: the whole matrix is tail (no one-thread-per-row head)."""
    n = 5003
    rng = np.random.default_rng(11)
    has = rng.random(n) < 0.6
    rp = np.zeros(n + 1, np.int64)
    np.cumsum(has, out=rp[1:])
    col = rng.integers(0, n, int(has.sum())).astype(np.int32)
    csr = CSR(n, rp.astype(np.int32), col, rng.integers(-8, 9, col.size).astype(np.float64))
    x = rng.integers(-8, 9, n).astype(np.float64)
    with build(csr, "sell", C=32, sigma=1 << 30) as A:
        d = A.describe()
        assert d["tail_positions"] == d["n_slices"] * 32
        y = run(A, x)
        assert_parity(y, oracle.spmv(csr, x), np.float64, exact=True, label="unit rows")
        assert not np.signbit(y[~has]).any() and np.all(y[~has] == 0)


@pytest.mark.parametrize("spl", [1, 2, 4])
@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_gather_probe(dtype, spl):
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    tdt = torch.float64 if dtype == np.float64 else torch.float32
    code = 0 if dtype == np.float64 else 1
    x = torch.ones(1 << 20, dtype=tdt, device="cuda")
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    done = spmv.spmv_probe_gather(x, x.numel(), code, spl, 1 << 22, out)
    torch.cuda.synchronize()
    assert done >= 1 << 22
    assert out.item() == done  # every gathered value is 1, so the sum counts the lane loads
    if spl > 1:  # x of exactly one line: every lane load stays inside it
        one = torch.ones(128 // x.element_size(), dtype=tdt, device="cuda")
        out.zero_()
        done = spmv.spmv_probe_gather(one, one.numel(), code, spl, 1 << 20, out)
        torch.cuda.synchronize()
        assert out.item() == done
        with pytest.raises(spmv.SpmvError):  # less than one line
            spmv.spmv_probe_gather(one, one.numel() - 1, code, spl, 10, out)
    with pytest.raises(spmv.SpmvError):
        spmv.spmv_probe_gather(x, 0, code, spl, 10, out)
    with pytest.raises(spmv.SpmvError):
        spmv.spmv_probe_gather(x, x.numel(), code, 3, 10, out)


def test_device_status_after_staged_applies():
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    csr = _tail_matrix(4099, seed=1, dtype=np.float64, integer=True)
    x = np.random.default_rng(2).integers(-8, 9, csr.n).astype(np.float64)
    with build(csr, "sell", staged=1) as A:
        assert A.describe()["staged"]
        for _ in range(3):
            y = run(A, x)
        spmv.spmv_device_status(A._h)  # raises SPMV_ERR_TIMEOUT if a bounded wait ran out
        assert_parity(y, oracle.spmv(csr, x), np.float64, exact=True, label="staged")


@pytest.mark.parametrize("shape", ["1d", "2d"])
def test_width_exact_kernel_above_a_wave(shape):
    """Float64 matrices whose longest row is 3 or 5 entries, with more row positions than
    one wave of threads (152 x 2048), take the width-exact kernel at 6 CTAs per SM."""
    from workloads import integer_x, laplacian_1d, laplacian_2d

    csr = laplacian_1d(400_003) if shape == "1d" else laplacian_2d(601, 599)
    assert csr.n > 152 * 2048
    for integer in (True, False):
        x = integer_x(csr.n) if integer else uniform_x(csr.n)
        with build(csr, "auto") as A:
            d = A.describe()
            assert d["format"] == "sell" and d["max_width"] in (3, 5) and d["sigma"] == 1
            y = run(A, x)
            assert_parity(y, oracle.spmv(csr, x), np.float64, exact=integer, label=f"{shape} integer={integer}")


@pytest.mark.parametrize("integer", [True, False], ids=["integer", "real"])
def test_capped_tail_loops_without_long_rows(integer):
    """No row longer than the threshold, so no chunks share the launch: the tail runs on
    at most 12 CTAs per SM, each looping over groups of 64 rows.  2.5 M rows, three in
    four of at most 2 entries, give over two groups per warp."""
    from workloads import CSR

    rng = np.random.default_rng(31)
    n = 2_500_000
    lens = rng.choice([0, 1, 2, 3, 7], size=n, p=[0.15, 0.45, 0.25, 0.1, 0.05])
    rp = np.zeros(n + 1, np.int64)
    np.cumsum(lens, out=rp[1:])
    col = rng.integers(2, n, size=int(rp[-1])).astype(np.int32)  # unsorted, duplicates allowed
    vals = (rng.integers(-8, 9, col.size) if integer else rng.standard_normal(col.size)).astype(np.float64)
    csr = CSR(n, rp.astype(np.int32), col, vals)
    x = (rng.integers(-8, 9, n) if integer else uniform_x(n, seed=32)).astype(np.float64)
    x[0], x[1] = np.inf, np.nan  # referenced by no stored entry
    with build(csr, "sell", C=32, sigma=1 << 30) as A:
        d = A.describe()
        assert d["n_long_rows"] == 0 and d["tail_positions"] > 12 * 152 * 8 * 64, d
        y = run(A, x)
        assert np.all(np.isfinite(y))
        assert_parity(y, oracle.spmv(csr, x), np.float64, exact=integer, label="capped tail")
