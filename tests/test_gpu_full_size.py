"""Parity at the full workload sizes, in the launch configuration the bench times (AUTO format).

The oracle evaluates sampled rows one by one (random rows, both ends, every long row); the
Laplacians are also checked on every row against their closed forms, and the 2D Laplacian
bit-exactly on integer x.  Each tolerance check records its worst error ratio,
|y - y_ref| / (tau * sum |a_ij x_j|) over the checked rows, as the test property
``worst_error_ratio`` and on a ``worst error ratio`` output line.
"""
import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_parity, build, run
from workloads import integer_x, make_workload

pytestmark = pytest.mark.gpu


def record_worst(record_property, label, worst):
    record_property("worst_error_ratio", worst)
    print(f"worst error ratio {label}: {worst:.3e}")


def sample_rows(csr, k=20000, seed=0, extra=()):
    rng = np.random.default_rng(seed)
    n = csr.n
    rows = np.concatenate([np.arange(min(n, 1000)), np.arange(max(0, n - 1000), n),
                           rng.integers(0, n, size=min(k, n)), np.asarray(extra, dtype=np.int64)])
    return np.unique(rows)


def stencil_expect(grid, f):
    """y of the Dirichlet Laplacian applied to x = f(position): missing neighbours contribute f there."""
    dims = len(grid)
    idx = np.arange(int(np.prod(grid)), dtype=np.int64)
    coords, rest = [], idx
    for g in grid:
        coords.append(rest % g)
        rest = rest // g
    y = np.zeros(idx.size)
    for axis in range(dims):
        for step in (-1, 1):
            q = [c.copy() for c in coords]
            q[axis] = q[axis] + step
            missing = (q[axis] < 0) | (q[axis] >= grid[axis])
            y[missing] += f(*q)[missing]
    return y


@pytest.mark.parametrize("name,dtype", [("lap3d_128", np.float64), ("lap3d_128", np.float32),
                                        ("hmep_6p2m", np.float64), ("powerlaw_4m", np.float64),
                                        ("uniform16_16m", np.float32), ("lap2d_256", np.float64)])
def test_full_size_sampled_rows(name, dtype, record_property):
    csr, x = make_workload(name, dtype=dtype)
    extra = []
    if name.startswith("powerlaw"):
        lens = np.diff(csr.row_ptr.astype(np.int64))
        # long rows go to the row-split chunks: a spread of 2000 of them over the whole
        # matrix, and every one of the 32 dense rows (200k - 1M entries, hundreds of chunks)
        long_rows = np.nonzero(lens > 128)[0]
        dense = np.argsort(-lens, kind="stable")[:32]
        assert lens[dense].min() >= 200_000
        extra = np.concatenate([long_rows[np.linspace(0, long_rows.size - 1, 2000).astype(np.int64)], dense])
    rows = sample_rows(csr, extra=extra)
    ref = oracle.spmv(csr, x, rows=rows)
    with build(csr, "auto") as A:
        y = run(A, x)
        assert np.all(np.isfinite(y))
        label = f"{name} {np.dtype(dtype).name} ({A.describe()['format']})"
        record_worst(record_property, label, assert_parity(y[rows], ref, dtype, label=label))


@pytest.mark.parametrize("fmt,params", [("csr_vector", {}), ("ell_r", {}), ("sell", {"C": 64, "sigma": 256}),
                                        ("hyb", {}), ("hyb", {"spill_csr": 0}), ("merge", {})])
def test_full_size_uniform_every_format(fmt, params, record_property):
    """The random uniform workload is the one swept over every format."""
    csr, x = make_workload("uniform16_16m")
    rows = sample_rows(csr, k=5000, seed=1)
    ref = oracle.spmv(csr, x, rows=rows)
    with build(csr, fmt, **params) as A:
        label = f"uniform16_16m float32 ({fmt} {params})"
        record_worst(record_property, label, assert_parity(run(A, x)[rows], ref, np.float32, label=label))


@pytest.mark.parametrize("fmt", ["merge", "hyb", "csr_vector"])
def test_full_size_powerlaw_other_formats(fmt, record_property):
    csr, x = make_workload("powerlaw_4m")
    lens = np.diff(csr.row_ptr.astype(np.int64))
    rows = sample_rows(csr, k=5000, seed=2, extra=np.argsort(-lens)[:64])
    ref = oracle.spmv(csr, x, rows=rows)
    with build(csr, fmt) as A:
        label = f"powerlaw_4m float64 ({fmt})"
        record_worst(record_property, label, assert_parity(run(A, x)[rows], ref, np.float64, label=label))


def test_full_size_laplacian_closed_forms():
    """Every row of the full-size Laplacians against the closed form (exact integers)."""
    for name, grid, (a, b, c, d) in [("lap3d_128", (128, 128, 128), (1, -2, 3, 5)),
                                     ("lap2d_256", (256, 256), (3, -1, 0, 7))]:
        csr, _ = make_workload(name)
        coords, rest = [], np.arange(csr.n, dtype=np.int64)
        for g in grid:
            coords.append(rest % g)
            rest = rest // g
        coef = (a, b, c)[:len(grid)]
        x = (sum(k * q for k, q in zip(coef, coords)) + d).astype(np.float64)
        expect = stencil_expect(grid, lambda *q: sum(k * v for k, v in zip(coef, q)) + d)
        with build(csr, "auto") as A:
            y = run(A, x)
        assert np.array_equal(y, expect), name


def test_full_size_integer_x_bit_exact():
    csr, _ = make_workload("lap2d_256")
    x = integer_x(csr.n)
    ref = oracle.spmv(csr, x)
    with build(csr, "auto") as A:
        assert_parity(run(A, x), ref, np.float64, exact=True, label="lap2d_256 integer x")


# --------------------------------------------------------------------------- #
# maximum sizes: more than 2^31 slots (64-bit slot offsets in the fill, the apply
# and the round trip), integer data, every row compared bit for bit
# --------------------------------------------------------------------------- #


def _wide_rows_matrix(n, long_every, long_len, seed):
    """n rows of one entry each, except every `long_every`-th row (and the last) with
    `long_len` distinct sorted columns; integer values in [-3, 3]."""
    from workloads import CSR

    rng = np.random.default_rng(seed)
    lens = np.ones(n, np.int64)
    lens[::long_every] = long_len
    lens[-1] = long_len
    row_ptr = np.zeros(n + 1, np.int64)
    np.cumsum(lens, out=row_ptr[1:])
    cols = rng.integers(0, n, size=int(row_ptr[-1]), dtype=np.int32)
    long_rows = np.nonzero(lens == long_len)[0]
    # distinct inside a row: 6007 is odd, so j -> 6007 j is one-to-one modulo n = 2^k
    base = np.sort((long_rows[:, None] * 7919 + np.arange(long_len)[None, :] * 6007) % n, axis=1)
    cols[(row_ptr[long_rows][:, None] + np.arange(long_len)[None, :]).ravel()] = base.ravel()
    vals = rng.integers(-3, 4, size=cols.size, dtype=np.int8).astype(np.float64)
    return CSR(n, row_ptr.astype(np.int32), cols.astype(np.int32), vals)


@pytest.mark.parametrize("fmt,params,long_every", [
    ("ell_r", {"long_row_threshold": 0}, 1 << 21),
    ("ell_r", {"long_row_threshold": 0, "row_threads": 4}, 1 << 21),
    ("sell", {"C": 64, "sigma": 1, "long_row_threshold": 0}, 64),
])
def test_more_than_2_31_slots(fmt, params, long_every):
    n, long_len = 1 << 22, 600
    csr = _wide_rows_matrix(n, long_every, long_len, seed=11)
    x = integer_x(n, seed=12)
    with build(csr, fmt, **params) as A:
        d = A.describe()
        assert d["slots"] > 2 ** 31, d["slots"]
        y = run(A, x)
        assert_parity(y, oracle.spmv(csr, x), np.float64, exact=True, label=f"{fmt} {params}")
