"""Applies of ONE handle on two streams at once.

The apply only reads the handle; the arrays it writes besides y (merge-path and COO
carries, row-split partials and counters, the scratch column of a scaled apply
without a fused epilogue, the host-apply staging) are kept once per stream.  Each
case enqueues many applies alternately on two non-blocking streams, each stream with
its own x and y, with no synchronisation in between, so kernels of the two streams
overlap on the GPU.  Both results must match the oracle: within the per-row tolerance
on real-valued data, bit for bit on integer-valued data.
"""
import threading

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_parity, build, torch_cuda
from workloads import CSR, integer_x, make_workload, uniform_x

pytestmark = pytest.mark.gpu

#: plans that write scratch during the apply (each asserted below)
PLANS = [
    ("auto", {}, "row-split"),                       # sorted SELL + long-row chunks in one launch
    ("hyb", {}, "COO spill"),                        # ELL part + load-balanced COO spill + carries
    ("hyb", {"spill_csr": 1}, "CSR spill"),          # ELL part + merge-path spill + carries
    ("merge", {}, "merge-path"),                     # merge-path over every row + carries
    ("csr_vector", {}, "csr-vector + row-split"),    # length bins, long rows to the row-split pass
]


def _matrix(integer):
    csr, _ = make_workload("powerlaw_small")
    if integer:
        rng = np.random.default_rng(21)
        csr = CSR(csr.n, csr.row_ptr, csr.col_idx, rng.integers(-8, 9, csr.nnz).astype(np.float64))
    return csr


def _vectors(n, integer):
    if integer:
        return integer_x(n, seed=102), integer_x(n, seed=103)
    return uniform_x(n, seed=101), uniform_x(n, seed=104)


def _uses_scratch(d, label):
    if label.startswith("csr-vector") or label == "row-split":
        assert d["n_long_rows"] > 0, d
    else:
        assert d["segment"] != "none" and d["segment_ctas"] > 1, d


@pytest.mark.parametrize("integer", [False, True], ids=["real", "integer"])
@pytest.mark.parametrize("plan", PLANS, ids=[p[2] for p in PLANS])
def test_two_streams_one_handle(plan, integer):
    torch = torch_cuda()
    fmt, params, label = plan
    csr = _matrix(integer)
    xa_np, xb_np = _vectors(csr.n, integer)
    with build(csr, fmt, **params) as A:
        _uses_scratch(A.describe(), label)
        xa, xb = torch.from_numpy(xa_np).cuda(), torch.from_numpy(xb_np).cuda()
        ya, yb = torch.full_like(xa, float("nan")), torch.full_like(xb, float("nan"))
        sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
        torch.cuda.synchronize()
        for _ in range(40):
            A.apply(xa, ya, stream=sa)
            A.apply(xb, yb, stream=sb)
        torch.cuda.synchronize()
        for x_np, y, tag in ((xa_np, ya, "stream a"), (xb_np, yb, "stream b")):
            assert_parity(y.cpu().numpy(), oracle.spmv(csr, x_np), np.float64, exact=integer,
                          label=f"{label} {tag}")


@pytest.mark.parametrize("plan", [p for p in PLANS if p[0] != "auto"], ids=[p[2] for p in PLANS if p[0] != "auto"])
def test_two_streams_scaled_apply(plan):
    """y = 2 A x + 0.5 y goes through a scratch column on these formats (no fused epilogue)."""
    import sparse_matrix_vector_csr_gb300 as spmv

    torch = torch_cuda()
    fmt, params, label = plan
    csr = _matrix(True)
    xa_np, xb_np = _vectors(csr.n, True)
    y0a, y0b = integer_x(csr.n, seed=201), integer_x(csr.n, seed=202)
    with build(csr, fmt, **params) as A:
        xa, xb = torch.from_numpy(xa_np).cuda(), torch.from_numpy(xb_np).cuda()
        sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
        ya, yb = torch.from_numpy(y0a).cuda(), torch.from_numpy(y0b).cuda()
        torch.cuda.synchronize()
        for _ in range(10):  # y <- 2 A x + 0.5 y, ten times on each stream, interleaved
            spmv.spmv_apply_ex(A._h, 2.0, xa, 0.5, ya, sa)
            spmv.spmv_apply_ex(A._h, 2.0, xb, 0.5, yb, sb)
        torch.cuda.synchronize()
        for x_np, y0, y, tag in ((xa_np, y0a, ya, "a"), (xb_np, y0b, yb, "b")):
            ax = oracle.spmv(csr, x_np)["y_hi"]
            want = y0.copy()
            for _ in range(10):
                want = 2.0 * ax + 0.5 * want
            got = y.cpu().numpy()
            # integer A x; 0.5 y halves exactly while the values stay far from the last bit
            assert np.array_equal(got, want), f"{label} stream {tag}: first mismatch at {np.argmax(got != want)}"


@pytest.mark.parametrize("plan", PLANS[:2], ids=[p[2] for p in PLANS[:2]])
def test_two_host_threads_apply_host(plan):
    """Two host threads call spmv_apply_host on one handle with their own streams."""
    torch = torch_cuda()
    fmt, params, label = plan
    csr = _matrix(True)
    xs = _vectors(csr.n, True)
    results, errors = [None, None], []
    with build(csr, fmt, **params) as A:
        def worker(i):
            try:
                torch.cuda.set_device(0)
                s = torch.cuda.Stream()
                xh = torch.from_numpy(xs[i]).pin_memory().numpy()
                yh = torch.empty(csr.n, dtype=torch.float64).pin_memory().numpy()
                for _ in range(20):
                    A.apply_host(xh, yh, stream=s)
                results[i] = yh.copy()
            except Exception as e:  # reported in the main thread
                errors.append(e)

        threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
    assert not errors, errors
    for i in range(2):
        assert_parity(results[i], oracle.spmv(csr, xs[i]), np.float64, exact=True, label=f"{label} thread {i}")


@pytest.mark.parametrize("plan", PLANS, ids=[p[2] for p in PLANS])
def test_first_apply_inside_a_capture(plan):
    """The first apply of a handle on a stream is captured into a graph, so the stream's
    scratch set is allocated then.  An apply enqueued on that stream outside the graph
    before the graph has ever run, then replays of the graph, then another apply outside
    it, all match the oracle bit for bit."""
    torch = torch_cuda()
    fmt, params, label = plan
    csr = _matrix(True)
    xa_np, xb_np = _vectors(csr.n, True)
    want_a, want_b = oracle.spmv(csr, xa_np), oracle.spmv(csr, xb_np)
    with build(csr, fmt, **params) as A:
        _uses_scratch(A.describe(), label)
        xa, xb = torch.from_numpy(xa_np).cuda(), torch.from_numpy(xb_np).cuda()
        ya, yb = torch.full_like(xa, float("nan")), torch.full_like(xb, float("nan"))
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            A.apply(xa, ya, stream=s)
        with torch.cuda.stream(s):
            A.apply(xb, yb, stream=s)  # the graph has not run yet
        s.synchronize()
        assert_parity(yb.cpu().numpy(), want_b, np.float64, exact=True, label=f"{label} outside the graph")
        for _ in range(3):
            ya.fill_(float("nan"))
            with torch.cuda.stream(s):
                g.replay()
            s.synchronize()
            assert_parity(ya.cpu().numpy(), want_a, np.float64, exact=True, label=f"{label} graph replay")
        yb.fill_(float("nan"))
        with torch.cuda.stream(s):
            A.apply(xb, yb, stream=s)
        s.synchronize()
        assert_parity(yb.cpu().numpy(), want_b, np.float64, exact=True, label=f"{label} after the replays")
        del g
