"""GPU parity: the CUDA path against the oracle, element by element, through the C ABI.

Acceptance rule (per row i):  |y_gpu - y_ref| <= tau * sum_j |a_ij x_j| with
tau = 1e-12 for float64 and 1e-5 for float32, y_ref the long double oracle value;
bit-exact equality on integer-valued matrices and vectors, where every partial
sum is an exactly representable integer whatever the summation order.
"""
import numpy as np
import pytest

import oracle
from oracle import layout
from tests.gpu_util import (FORMAT_CASES, assert_parity, assert_roundtrip, build, case_id, run,
                            torch_cuda)
from workloads import CSR, laplacian_2d, make_workload, random_csr, integer_x, uniform_x

pytestmark = pytest.mark.gpu

SMALL = ["lap2d_small", "lap3d_small", "hmep_small", "powerlaw_small", "uniform16_small", "band_small"]

_cache = {}


def small(name, dtype=None):
    key = (name, dtype)
    if key not in _cache:
        csr, x = make_workload(name, dtype=dtype)
        _cache[key] = (csr, x, oracle.spmv(csr, x))
    return _cache[key]


@pytest.mark.parametrize("case", FORMAT_CASES, ids=case_id)
@pytest.mark.parametrize("name", SMALL)
def test_small_workloads_all_formats(name, case):
    fmt, params = case
    csr, x, ref = small(name)
    with build(csr, fmt, **params) as A:
        y = run(A, x)
        assert_parity(y, ref, csr.dtype, label=f"{name}/{case_id(case)}")
        assert_roundtrip(A, csr, label=f"{name}/{case_id(case)}")


@pytest.mark.parametrize("case", [c for c in FORMAT_CASES if c[0] in ("auto", "csr_vector", "sell", "hyb", "merge")],
                         ids=case_id)
@pytest.mark.parametrize("name", ["lap3d_small", "powerlaw_small", "hmep_small"])
def test_small_workloads_float32(name, case):
    fmt, params = case
    csr, x, ref = small(name, np.float32)
    with build(csr, fmt, **params) as A:
        y = run(A, x)
        assert_parity(y, ref, np.float32, label=f"{name}/f32/{case_id(case)}")
        assert_roundtrip(A, csr)


@pytest.mark.parametrize("case", FORMAT_CASES, ids=case_id)
@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_integer_inputs_bit_exact(case, dtype):
    fmt, params = case
    A_csr = laplacian_2d(256, 256, dtype=dtype)
    x = integer_x(A_csr.n, dtype=dtype)
    ref = oracle.spmv(A_csr, x)
    with build(A_csr, fmt, **params) as A:
        assert_parity(run(A, x), ref, dtype, exact=True, label=f"lap2d_256 integer x/{case_id(case)}")
    R = random_csr(3000, 0.004, seed=7, dtype=dtype, integer_values=True, duplicates=True, unsorted=True,
                   empty_row_fraction=0.2, full_rows=2)
    xr = integer_x(R.n, seed=3, dtype=dtype)
    ref = oracle.spmv(R, xr)
    with build(R, fmt, **params) as A:
        assert_parity(run(A, xr), ref, dtype, exact=True, label=f"random integer/{case_id(case)}")
        assert_roundtrip(A, R)


@pytest.mark.parametrize("case", FORMAT_CASES, ids=case_id)
def test_duplicates_unsorted_empty_rows(case):
    fmt, params = case
    for seed in (1, 2):
        csr = random_csr(2500, 0.01, seed=seed, duplicates=True, unsorted=True, empty_row_fraction=0.3, full_rows=1)
        x = uniform_x(csr.n, seed=seed)
        with build(csr, fmt, **params) as A:
            assert_parity(run(A, x), oracle.spmv(csr, x), np.float64, label=case_id(case))
            assert_roundtrip(A, csr)


# --------------------------------------------------------------------------- #
# degenerate and extreme shapes
# --------------------------------------------------------------------------- #


def _csr_from_rows(n, rows, dtype=np.float64, seed=0, integer=False):
    rng = np.random.default_rng(seed)
    lens = np.array([len(r) for r in rows], dtype=np.int64)
    rp = np.zeros(n + 1, np.int64)
    np.cumsum(lens, out=rp[1:])
    col = np.concatenate([np.asarray(r, np.int64) for r in rows]).astype(np.int32) if lens.sum() else np.zeros(0, np.int32)
    vals = (rng.integers(-8, 9, col.size) if integer else rng.standard_normal(col.size)).astype(dtype)
    return CSR(n, rp.astype(np.int32), col, vals)


@pytest.mark.parametrize("case", FORMAT_CASES, ids=case_id)
def test_all_rows_empty(case):
    fmt, params = case
    n = 1000
    csr = CSR(n, np.zeros(n + 1, np.int32), np.zeros(0, np.int32), np.zeros(0, np.float64))
    with build(csr, fmt, **params) as A:
        y = run(A, uniform_x(n))
        assert np.all(y == 0) and not np.any(np.signbit(y))


def test_zero_order_matrix():
    torch = torch_cuda()
    csr = CSR(0, np.zeros(1, np.int32), np.zeros(0, np.int32), np.zeros(0, np.float64))
    with build(csr, "auto") as A:
        x = torch.zeros(0, dtype=torch.float64, device="cuda")
        A.apply(x, torch.zeros(0, dtype=torch.float64, device="cuda"))
        assert A.describe()["n"] == 0


@pytest.mark.parametrize("fmt", ["auto", "csr_vector", "sell", "hyb", "merge"])
@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_single_row_of_a_million(fmt, dtype):
    """One row with 10^6 entries spread over several hundred work units (merge-path CTAs or
    row-split chunks)."""
    n = 1_000_000
    row_ptr = np.full(n + 1, n, dtype=np.int32)
    row_ptr[0] = 0
    rng = np.random.default_rng(5)
    for integer in (True, False):
        vals = (rng.integers(-8, 9, n) if integer else rng.standard_normal(n)).astype(dtype)
        csr = CSR(n, row_ptr, np.arange(n, dtype=np.int32), vals)
        x = integer_x(n, dtype=dtype) if integer else uniform_x(n, dtype=dtype)
        ref = oracle.spmv(csr, x, rows=np.arange(0, n, 997))
        with build(csr, fmt) as A:
            y = run(A, x)
            d = A.describe()
            # hundreds of work units: merge-path shares of 2048 items, or row-split chunks
            # of 4096 (float64) / 2048 (float32) entries
            assert d["segment"] != "none" and d["segment_ctas"] >= 240
            assert_parity(y[::997], ref, dtype, exact=integer, label=f"{fmt} integer={integer}")


@pytest.mark.parametrize("case", FORMAT_CASES, ids=case_id)
def test_alternating_empty_and_long_rows(case):
    fmt, params = case
    n = 20000
    rng = np.random.default_rng(3)
    rows = [np.sort(rng.choice(n, 5000, replace=False)) if i % 2 == 0 and i < 40 else
            (np.sort(rng.choice(n, 3, replace=False)) if i % 3 == 0 else []) for i in range(n)]
    for integer in (True, False):
        csr = _csr_from_rows(n, rows, seed=4, integer=integer)
        x = integer_x(n) if integer else uniform_x(n)
        with build(csr, fmt, **params) as A:
            assert_parity(run(A, x), oracle.spmv(csr, x), np.float64, exact=integer, label=case_id(case))
            assert_roundtrip(A, csr)


@pytest.mark.parametrize("case", FORMAT_CASES, ids=case_id)
def test_padding_never_touches_x(case):
    """x is +Inf and NaN at columns no stored entry uses; padding must not pick them up."""
    fmt, params = case
    n = 4096
    rng = np.random.default_rng(9)
    rows = [np.sort(rng.choice(np.arange(2, n), rng.integers(0, 40), replace=False)) for _ in range(n)]
    csr = _csr_from_rows(n, rows, seed=2)
    x = uniform_x(n)
    x[0], x[1] = np.inf, np.nan
    with build(csr, fmt, **params) as A:
        y = run(A, x)
        assert np.all(np.isfinite(y))
        assert_parity(y, oracle.spmv(csr, x), np.float64, label=case_id(case))


# --------------------------------------------------------------------------- #
# layouts against the oracle's layout definitions (bit-exact integer work)
# --------------------------------------------------------------------------- #


@pytest.mark.parametrize("C,sigma", [(32, 1), (32, 256), (64, 1), (64, 2048), (32, 4096), (32, 1 << 30)])
@pytest.mark.parametrize("name", ["powerlaw_small", "hmep_small", "lap3d_small"])
def test_sell_layout_matches_definition(name, C, sigma):
    csr, _, _ = small(name)
    lens = layout.row_lengths(csr.row_ptr)
    with build(csr, "sell", C=C, sigma=sigma) as A:
        d = A.describe()
        thr = d["long_row_threshold"]
        exp = layout.sell_layout(lens, C, min(sigma, csr.n), exclude=layout.long_rows(lens, thr))
        perm, sp = A.layout()
        assert np.array_equal(perm.cpu().numpy(), exp["perm"])
        assert np.array_equal(sp.cpu().numpy(), exp["slice_ptr"])
        assert d["padded_entries"] == exp["padded_entries"]
        assert d["slots"] == exp["allocated_slots"]
        assert d["n_long_rows"] == layout.long_rows(lens, thr).size


SLOT_CASES = [("sell", 32, 1, 1, 0), ("sell", 64, 256, 1, 0), ("sell", 32, 1, 4, 1), ("sell", 32, 1 << 30, 8, 1),
              ("sell", 64, 1, 8, 0), ("sell", 32, 4096, 32, 1), ("ell_r", 0, 1, 1, 0), ("ell_r", 0, 1, 4, 1),
              ("ell_r", 0, 1, 2, 0), ("sell", 32, 1, 4, 2), ("ell_r", 0, 1, 8, 2),
              ("sell", 32, 1, 1, "vec"), ("sell", 64, 1 << 30, 1, "vec"), ("ell_r", 0, 1, 1, "vec")]


@pytest.mark.parametrize("fmt,C,sigma,g,il", SLOT_CASES, ids=[f"{f}-C{c}-s{s}-g{g}-i{i}" for f, c, s, g, i in SLOT_CASES])
@pytest.mark.parametrize("name", ["powerlaw_small", "hmep_small", "lap3d_small"])
def test_slot_arrays_match_definition(name, fmt, C, sigma, g, il):
    """Every slot of the sliced part (column and value, padding included) against the
    oracle's layout definition: bit-exact index and byte work."""
    csr, _, _ = small(name)
    lens = layout.row_lengths(csr.row_ptr)
    vec = il == "vec"
    kw = {"row_threads": g, "row_group_mode": 0 if vec else il, "vector_loads": 1 if vec else 0}
    if fmt == "sell":
        kw.update(C=C, sigma=sigma)
    with build(csr, fmt, **kw) as A:
        d = A.describe()
        assert d["row_threads"] == g and d["vector_loads"] == int(vec)
        exclude = layout.long_rows(lens, d["long_row_threshold"])
        if vec:  # indices in 4s, values in 16-byte groups, widths a multiple of 4
            opts = dict(group=4, interleaved=True, group_val=16 // csr.vals.dtype.itemsize, round_to=4)
        else:
            assert d["row_group_mode"] == il
            opts = dict(group=g, interleaved=il == 1)
        if fmt == "sell":
            exp = layout.sell_slots(csr, C, min(sigma, csr.n), exclude=exclude, **opts)
        else:
            exp = layout.sell_slots(csr, 0, 1, exclude=exclude, ell_ld=d["ld"], **opts)
        col, val = A.slots()
        assert col.numel() == exp[0].size == d["slots"]
        assert np.array_equal(col.cpu().numpy(), exp[0])
        assert np.array_equal(val.cpu().numpy().view(np.uint8), exp[1].view(np.uint8))


@pytest.mark.parametrize("N,b_r", [(1024, 32), (4096, 32), (4096, 64), (777, 64)])
def test_pjds_storage_of_one_full_row(N, b_r):
    """One full row + one entry per other row: pJDS stores (b_r + 1) N - b_r, ELLPACK N^2."""
    rows = [[i % N] for i in range(N)]
    rows[N // 3] = list(range(N))
    csr = _csr_from_rows(N, rows)
    with build(csr, "sell", C=b_r, sigma=1 << 30, long_row_threshold=0) as A:
        assert A.describe()["padded_entries"] == (b_r + 1) * N - b_r
    with build(csr, "ell_r", long_row_threshold=0) as A:
        d = A.describe()
        assert d["padded_entries"] == N * N
        assert d["ld"] % 32 == 0 and d["ld"] >= N


@pytest.mark.parametrize("name", ["powerlaw_small", "hmep_small", "uniform16_small"])
@pytest.mark.parametrize("dtype", [np.float64, np.float32])
def test_hyb_split_matches_rule(name, dtype):
    csr, x, _ = small(name)
    csr = csr.astype(dtype)
    x = x.astype(dtype)
    lens = layout.row_lengths(csr.row_ptr)
    vb = np.dtype(dtype).itemsize
    ld = layout.ell_leading_dim(csr.n)
    cap = 4096 if dtype == np.float64 else 128
    K = layout.hyb_width(lens, vb, ld, c=4.0, k_cap=cap)  # each spilled entry's bytes weighted 4 against a streamed ELL slot's
    split = layout.hyb_split(lens, K)
    with build(csr, "hyb") as A:
        d = A.describe()
        assert d["K"] == K and d["ld"] == ld and d["ld"] % 256 == 0
        assert d["segment_nnz"] == split["spill_nnz"]
        assert d["segment_rows"] == split["spill_rows"].size
        assert_parity(run(A, x), oracle.spmv(csr, x), dtype)


def test_csr_vector_bins():
    csr, _, _ = small("powerlaw_small")
    lens = layout.row_lengths(csr.row_ptr)
    with build(csr, "csr_vector") as A:
        d = A.describe()
        thr = d["long_row_threshold"]
        short = lens[lens <= thr]
        # about eight entries a lane: 2 lanes up to 16 entries, then 4, 8, 16 up to 32, 64, 128, 32 above
        expect = {2: (short <= 16).sum(), 4: ((short > 16) & (short <= 32)).sum(), 8: ((short > 32) & (short <= 64)).sum(),
                  16: ((short > 64) & (short <= 128)).sum(), 32: (short > 128).sum()}
        got = {g: c for g, c in d["bins"]}
        assert got == {g: int(c) for g, c in expect.items() if c}
        assert d["n_long_rows"] == int((lens > thr).sum())


# --------------------------------------------------------------------------- #
# API behaviour
# --------------------------------------------------------------------------- #


def test_bad_csr_is_rejected():
    import sparse_matrix_vector_csr_gb300 as spmv

    good = random_csr(100, 0.05, seed=1)
    bad_cases = []
    c = good.col_idx.copy()
    c[3] = 100
    bad_cases.append(CSR(100, good.row_ptr, c, good.vals))
    r = good.row_ptr.copy()
    r[50], r[51] = r[51], r[50]
    if r[50] != r[51]:
        bad_cases.append(CSR(100, r, good.col_idx, good.vals))
    r2 = good.row_ptr.copy()
    r2[0] = 1
    bad_cases.append(CSR(100, r2, good.col_idx, good.vals))
    for bad in bad_cases:
        with pytest.raises(spmv.SpmvError) as ei:
            build(bad, "sell")
        assert ei.value.status == -2
    # the library still works afterwards
    x = uniform_x(100)
    with build(good, "sell") as A:
        assert_parity(run(A, x), oracle.spmv(good, x), np.float64)


def test_host_pointers_are_rejected():
    import sparse_matrix_vector_csr_gb300 as spmv

    csr = random_csr(50, 0.1, seed=1)
    with pytest.raises(spmv.SpmvError) as ei:
        spmv.spmv_build_from_csr(csr.n, csr.nnz, csr.row_ptr, csr.col_idx, csr.vals, 0, "sell")
    assert ei.value.status == -1


def test_host_vectors_are_refused_by_the_applies():
    """Vectors that are not device memory of the current device (a pageable numpy array,
    a pinned tensor) are refused before anything is enqueued; device vectors still work."""
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    csr = random_csr(300, 0.05, seed=4)
    x_np = uniform_x(csr.n)
    xd = torch.from_numpy(x_np).cuda()
    yd = torch.full_like(xd, float("nan"))
    pinned = torch.from_numpy(x_np.copy()).pin_memory()
    with build(csr, "auto") as A:
        h = A._h
        for bad_x, bad_y in ((x_np, yd), (xd, np.empty(csr.n)), (pinned, yd), (xd, pinned)):
            for call in (lambda: spmv.spmv_apply(h, bad_x, bad_y, 0),
                         lambda: spmv.spmv_apply_ex(h, 2.0, bad_x, 0.5, bad_y, 0),
                         lambda: spmv.spmv_permute_vector(h, bad_x, bad_y, 0, 0)):
                with pytest.raises(spmv.SpmvError) as ei:
                    call()
                assert ei.value.status == -1
        X = np.zeros((csr.n, 2))
        with pytest.raises(spmv.SpmvError) as ei:
            spmv.spmv_apply_multi(h, 2, 1.0, X, 2, 0.0, torch.zeros(csr.n, 2, dtype=torch.float64, device="cuda"), 2, 0)
        assert ei.value.status == -1
        with pytest.raises(spmv.SpmvError) as ei:
            spmv.spmv_cg(h, x_np, yd, 1e-8, 10, 0)
        assert ei.value.status == -1
        torch.cuda.synchronize()
        assert torch.isnan(yd).all()  # nothing ran
        A.apply(xd, yd)
        torch.cuda.synchronize()
        assert_parity(yd.cpu().numpy(), oracle.spmv(csr, x_np), np.float64)


def test_too_large_layout_is_refused():
    import sparse_matrix_vector_csr_gb300 as spmv

    n = 3_000_000
    rows_ptr = np.zeros(n + 1, np.int64)
    rows_ptr[1:] = n  # row 0 is full, the rest empty
    csr = CSR(n, rows_ptr.astype(np.int32), np.arange(n, dtype=np.int32), np.ones(n))
    with pytest.raises(spmv.SpmvError) as ei:
        build(csr, "ell_r", long_row_threshold=0)  # 3e6 x 3e6 rectangle
    assert ei.value.status == -5


def test_apply_on_a_side_stream_and_host_path():
    torch = torch_cuda()
    csr, x, ref = small("hmep_small")
    with build(csr, "auto") as A:
        s = torch.cuda.Stream()
        xd = torch.from_numpy(x).cuda()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            y = torch.empty_like(xd)
            A.apply(xd, y)
        s.synchronize()
        assert_parity(y.cpu().numpy(), ref, np.float64)
        xh = torch.from_numpy(x).pin_memory().numpy()
        yh = torch.empty(csr.n, dtype=torch.float64).pin_memory().numpy()
        A.apply_host(xh, yh)
        assert np.array_equal(yh, y.cpu().numpy())
        times = A.apply_profiled(xd, y)
        assert len(times) == len(A.describe()["kernels"]) and all(t > 0 for t in times)


def test_repeated_applies_are_deterministic():
    csr, x, _ = small("powerlaw_small")
    with build(csr, "sell", sigma=256) as A:
        y1 = run(A, x)
        y2 = run(A, x)
        assert np.array_equal(y1.view(np.uint64), y2.view(np.uint64))


@pytest.mark.parametrize("fmt,name", [("auto", "powerlaw_small"), ("auto", "lap3d_small"), ("merge", "powerlaw_small"),
                                      ("hyb", "hmep_small"), ("csr_vector", "powerlaw_small")])
def test_apply_inside_a_cuda_graph(fmt, name):
    """Applies captured in a CUDA graph (back to back, as a solver loop would) replay correctly,
    including with a new x copied into the captured buffer between replays."""
    torch = torch_cuda()
    csr, x0, ref0 = small(name)
    x1 = uniform_x(csr.n, seed=55)
    ref1 = oracle.spmv(csr, x1)
    with build(csr, fmt) as A:
        xd = torch.from_numpy(x0).cuda()
        y = torch.empty_like(xd)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            A.apply(xd, y)  # warm-up outside the capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(3):
                A.apply(xd, y)
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_parity(y.cpu().numpy(), ref0, np.float64, label=f"graph {fmt} {name} x0")
        xd.copy_(torch.from_numpy(x1).cuda())
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_parity(y.cpu().numpy(), ref1, np.float64, label=f"graph {fmt} {name} x1")


def test_apply_after_a_kernel_that_writes_x():
    """The sliced kernel may start before the previous kernel of the stream ends; it must still
    read the x that kernel wrote (and not overwrite y that kernel reads)."""
    torch = torch_cuda()
    csr, x0, _ = small("lap3d_small")
    with build(csr, "auto") as A:
        xd = torch.from_numpy(x0).cuda()
        y = torch.empty_like(xd)
        for k in range(5):
            xd.mul_(-0.5).add_(1.0)          # a kernel producing x
            A.apply(xd, y)                   # reads it
            z = y * 2.0                      # a kernel reading y
            A.apply(xd, y)                   # rewrites y with the same values
            torch.cuda.synchronize()
            ref = oracle.spmv(csr, xd.cpu().numpy())
            assert_parity(y.cpu().numpy(), ref, np.float64, label=f"round {k}")
            assert torch.equal(z, y * 2.0)


def test_csr_vector_bin_boundaries():
    """Rows whose lengths sit on every bin edge (16/17, 32/33, 64/65, 128/129) and on the
    long-row threshold (256/257): each lands in its bin, the rows above 256 go to the
    row-split pass, and the product matches the oracle (bit for bit on integers)."""
    from workloads import CSR

    torch = torch_cuda()
    rng = np.random.default_rng(71)
    lens = np.array([0, 1, 16, 17, 32, 33, 64, 65, 128, 129, 256, 257, 1000] * 40)
    rng.shuffle(lens)
    n = 4096
    lens = np.concatenate([lens, rng.integers(0, 9, n - lens.size)])
    row_ptr = np.zeros(n + 1, np.int64)
    np.cumsum(lens, out=row_ptr[1:])
    cols = np.concatenate([np.sort(rng.choice(n, size=l, replace=False)) for l in lens]).astype(np.int32)
    vals = rng.integers(-4, 5, cols.size).astype(np.float64)
    csr = CSR(n, row_ptr.astype(np.int32), cols, vals)
    x = rng.integers(-8, 9, n).astype(np.float64)
    with build(csr, "csr_vector") as A:
        d = A.describe()
        assert d["long_row_threshold"] == 256
        short = lens[lens <= 256]
        expect = {2: (short <= 16).sum(), 4: ((short > 16) & (short <= 32)).sum(),
                  8: ((short > 32) & (short <= 64)).sum(), 16: ((short > 64) & (short <= 128)).sum(),
                  32: (short > 128).sum()}
        assert {g: c for g, c in d["bins"]} == {g: int(c) for g, c in expect.items() if c}
        assert d["n_long_rows"] == int((lens > 256).sum())
        y = A.apply(torch.from_numpy(x).cuda())
        torch.cuda.synchronize()
        assert_parity(y.cpu().numpy(), oracle.spmv(csr, x), np.float64, exact=True, label="bin edges")
