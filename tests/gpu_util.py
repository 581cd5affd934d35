"""Helpers shared by the GPU parity tests: device copies, CUDA-path runs, oracle checks."""
import numpy as np

import oracle


def torch_cuda():
    import torch

    if not torch.cuda.is_available():
        raise RuntimeError("these tests need a CUDA GPU")
    return torch


def to_device(csr):
    torch = torch_cuda()
    return (torch.from_numpy(np.ascontiguousarray(csr.row_ptr)).cuda(),
            torch.from_numpy(np.ascontiguousarray(csr.col_idx)).cuda(),
            torch.from_numpy(np.ascontiguousarray(csr.vals)).cuda())


def build(csr, fmt="auto", **params):
    import sparse_matrix_vector_csr_gb300 as spmv

    rp, ci, vv = to_device(csr)
    return spmv.SpmvMatrix.from_csr(rp, ci, vv, format=fmt, **params)


def run(A, x_np):
    torch = torch_cuda()
    x = torch.from_numpy(np.ascontiguousarray(x_np)).cuda()
    y = torch.full_like(x, float("nan"))  # every output element must be written
    A.apply(x, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def assert_parity(y, ref, dtype, exact=False, label=""):
    ok, worst, idx = oracle.check_rows(y, ref, dtype, exact=exact)
    if not ok:
        raise AssertionError(
            f"{label}: {'bit mismatch' if exact else 'tolerance exceeded'} (worst ratio {worst:.3g}) at row {idx}: "
            f"got {y[idx]!r}, oracle {ref['y_hi'][idx]!r} + {ref['y_lo'][idx]!r}, scale {ref['scale'][idx]!r}")
    return worst


def assert_roundtrip(A, csr, label=""):
    rp, ci, vv = A.to_csr()
    rp, ci, vv = rp.cpu().numpy(), ci.cpu().numpy(), vv.cpu().numpy()
    assert np.array_equal(rp, csr.row_ptr), f"{label}: row_ptr differs"
    assert np.array_equal(ci, csr.col_idx), f"{label}: col_idx differs"
    assert np.array_equal(vv.view(np.uint8), np.ascontiguousarray(csr.vals).view(np.uint8)), f"{label}: vals differ"


#: (format, params) combinations every small workload is swept over
FORMAT_CASES = [
    ("auto", {}),
    ("csr_vector", {}),
    ("csr_vector", {"subwarp": 2}),
    ("csr_vector", {"subwarp": 32}),
    ("csr_vector", {"long_row_threshold": 8}),
    ("ell_r", {}),
    ("sell", {"C": 32, "sigma": 1}),
    ("sell", {"C": 32, "sigma": 256}),
    ("sell", {"C": 64, "sigma": 1}),
    ("sell", {"C": 64, "sigma": 1 << 30}),
    ("sell", {"C": 32, "sigma": 4096}),
    ("sell", {"C": 32, "sigma": 1, "long_row_threshold": 8}),
    ("hyb", {}),
    ("hyb", {"spill_csr": 0}),
    ("hyb", {"K": 20}),
    ("hyb", {"K": 3, "spill_csr": 0}),
    ("hyb", {"K": 0}),
    ("merge", {}),
    # G threads per row: interleaved slots, row-grouped and column-grouped
    ("sell", {"row_threads": 4}),
    ("sell", {"row_threads": 8, "row_group_mode": 0}),
    ("sell", {"row_threads": 4, "row_group_mode": 2}),
    ("sell", {"C": 64, "sigma": 256, "row_threads": 8, "row_group_mode": 2}),
    ("ell_r", {"row_threads": 2, "row_group_mode": 2}),
    ("sell", {"C": 64, "sigma": 1 << 30, "row_threads": 32}),
    ("sell", {"row_threads": 2, "long_row_threshold": 8}),
    ("ell_r", {"row_threads": 16}),
    ("hyb", {"row_threads": 4, "K": 3, "spill_csr": 0}),
    ("sell", {"row_threads": 1}),
    # one thread per row with 16-byte vector loads
    ("sell", {"vector_loads": 1}),
    ("sell", {"C": 64, "sigma": 1 << 30, "vector_loads": 1, "long_row_threshold": 8}),
    ("ell_r", {"vector_loads": 1}),
    ("hyb", {"vector_loads": 1, "K": 5}),
    # slots staged in shared memory by bulk copies
    ("sell", {"staged": 1}),
    ("sell", {"sigma": 1 << 30, "staged": 1}),
    ("sell", {"staged": 1, "long_row_threshold": 8}),
]


def case_id(case):
    fmt, p = case
    return fmt + ("-" + "-".join(f"{k}{v}" for k, v in p.items()) if p else "")
