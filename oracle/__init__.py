"""Oracle for the sparse matrix-vector product and its storage layouts.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product (``sparse_matrix_vector_csr_gb300``) never imports it,
and this package never imports the product: the two share no code.

Contents
--------
* :func:`spmv` -- y = A x from the CSR definition, single-threaded long double
  (``spmv_oracle.c``), with the per-row tolerance scale sum |a_ij x_j|.
* :mod:`oracle.layout` -- the storage-layout definitions the formats follow
  (sorted/padded row blocks of ELLPACK-R / pJDS / SELL-C-sigma, the HYB split).
* :func:`spmv_scaled`, :func:`spmm` -- y = alpha A x + beta y and its multi-vector
  form Y = alpha A X + beta Y, from the long double product above.
* :func:`check_rows` -- the acceptance rule for a computed y.
* :func:`omp_spmv` -- not an oracle: the plain OpenMP CSR product the bench reports as
  the multi-core CPU baseline (``csr_omp.c``).
* :mod:`oracle.cg` -- conjugate gradients (Hestenes-Stiefel) in float64 on the
  product above, for the solver built on the library.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(``tests/test_cg_oracle_pins.py`` for CG) against values the pages state, closed
forms, and brute force; none of them is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spmv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_spmv.so")
_lock = threading.Lock()
_lib = None


def build(out_path: str = _LIB_PATH, mutation: int = 0) -> str:
    """Compile the C oracle with gcc (no GPU involved).  Returns the library path."""
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", out_path, _SRC, "-lm"]
    if mutation:
        cmd.insert(1, f"-DORACLE_MUTATION={int(mutation)}")
    subprocess.run(cmd, check=True)
    return out_path


_OMP_SRC = os.path.join(_HERE, "csr_omp.c")
_OMP_PATH = os.path.join(_HERE, "libcsr_omp.so")
_omp = None


def build_omp(out_path: str = _OMP_PATH) -> str:
    """Compile the multi-core CPU baseline (gcc -fopenmp).  Returns the library path."""
    subprocess.run(["gcc", "-O3", "-fopenmp", "-std=c11", "-shared", "-fPIC", "-o", out_path, _OMP_SRC],
                   check=True)
    return out_path


def omp_spmv(csr, x, schedule: str = "static", threads: int = 0):
    """y = A x by the OpenMP CSR baseline (value-type sums, stored order).  Returns
    (y, threads used)."""
    global _omp
    with _lock:
        if _omp is None:
            if not os.path.exists(_OMP_PATH) or os.path.getmtime(_OMP_PATH) < os.path.getmtime(_OMP_SRC):
                build_omp()
            lib = ctypes.CDLL(_OMP_PATH)
            lib.csr_omp_spmv.restype = ctypes.c_int
            lib.csr_omp_spmv.argtypes = [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
            _omp = lib
    dt = np.dtype(csr.vals.dtype)
    x = np.ascontiguousarray(x, dtype=dt)
    y = np.empty(csr.n, dt)
    used = _omp.csr_omp_spmv(csr.n, csr.row_ptr.ctypes.data, csr.col_idx.ctypes.data if csr.nnz else None,
                             csr.vals.ctypes.data if csr.nnz else None, _dtype_code(dt), x.ctypes.data,
                             y.ctypes.data, 1 if schedule == "dynamic" else 0, int(threads))
    return y, int(used)


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_ldbl_mant_dig.restype = ctypes.c_int
    lib.oracle_spmv_csr.restype = ctypes.c_int
    lib.oracle_spmv_csr.argtypes = [
        ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
    ]
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
                build()
            _lib = _bind(_LIB_PATH)
    return _lib


def ldbl_mant_dig() -> int:
    return int(load().oracle_ldbl_mant_dig())


def _dtype_code(dt) -> int:
    dt = np.dtype(dt)
    if dt == np.float64:
        return 0
    if dt == np.float32:
        return 1
    raise TypeError(f"unsupported value type {dt}")


def spmv(csr, x, rows=None, lib=None) -> dict:
    """Evaluate y = A x (all rows, or the listed ``rows``) by the CSR definition.

    Returns a dict with ``y_hi``/``y_lo`` (the long double result as a double pair),
    ``y`` (rounded once to the value type), and ``scale`` (sum |a_ij x_j|).
    """
    lib = lib or load()
    dt = np.dtype(csr.vals.dtype)
    code = _dtype_code(dt)
    x = np.ascontiguousarray(x, dtype=dt)
    if x.shape != (csr.n,):
        raise ValueError("x must have length n")
    row_ptr = np.ascontiguousarray(csr.row_ptr, dtype=np.int32)
    col_idx = np.ascontiguousarray(csr.col_idx, dtype=np.int32)
    vals = np.ascontiguousarray(csr.vals)
    if rows is None:
        nrows = csr.n
        rows_arr = None
        rows_ptr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
        rows_ptr = rows_arr.ctypes.data
    y_hi = np.empty(nrows, np.float64)
    y_lo = np.empty(nrows, np.float64)
    scale = np.empty(nrows, np.float64)
    y = np.empty(nrows, dt)
    rc = lib.oracle_spmv_csr(
        csr.n, row_ptr.ctypes.data, col_idx.ctypes.data if col_idx.size else None,
        vals.ctypes.data if vals.size else None, code, x.ctypes.data if x.size else None,
        rows_ptr, nrows, y_hi.ctypes.data if nrows else None, y_lo.ctypes.data if nrows else None,
        scale.ctypes.data if nrows else None, y.ctypes.data if nrows else None)
    if rc != 0:
        raise ValueError("oracle rejected the CSR input (index out of range or non-monotone row_ptr)")
    return {"y_hi": y_hi, "y_lo": y_lo, "y": y, "scale": scale}


def spmv_scaled(csr, x, alpha, beta, y_old, rows=None, lib=None) -> dict:
    """y = alpha * A x + beta * y_old, combined in long double from the CSR result.

    beta == 0 does not read y_old (its content, NaN included, does not matter).  The
    tolerance scale becomes |alpha| * sum |a_ij x_j| + |beta * y_old_i|.
    """
    r = spmv(csr, x, rows=rows, lib=lib)
    dt = np.dtype(csr.vals.dtype)
    ax = r["y_hi"].astype(np.longdouble) + r["y_lo"].astype(np.longdouble)
    a = np.longdouble(alpha)
    if beta == 0:
        val = a * ax
        extra = np.zeros(ax.shape)
    else:
        yo = np.asarray(y_old, dtype=dt)
        if rows is not None:
            yo = yo[np.asarray(rows, dtype=np.int64)]
        val = a * ax + np.longdouble(beta) * yo.astype(np.longdouble)
        extra = np.abs(float(beta) * yo.astype(np.float64))
    hi = val.astype(np.float64)
    return {"y_hi": hi, "y_lo": (val - hi.astype(np.longdouble)).astype(np.float64), "y": val.astype(dt),
            "scale": abs(float(alpha)) * r["scale"] + extra}


def spmm(csr, X, alpha=1.0, beta=0.0, Y_old=None, rows=None, lib=None) -> dict:
    """Y = alpha * A X + beta * Y_old for the k columns of X (n x k), column by column.

    Returns the same keys as :func:`spmv_scaled`, each an array of shape (rows, k).
    """
    X = np.asarray(X)
    k = X.shape[1]
    cols = [spmv_scaled(csr, np.ascontiguousarray(X[:, c]), alpha, beta,
                        None if Y_old is None else np.ascontiguousarray(np.asarray(Y_old)[:, c]), rows=rows, lib=lib)
            for c in range(k)]
    return {key: np.stack([cc[key] for cc in cols], axis=1) for key in ("y_hi", "y_lo", "y", "scale")}


#: per-row tolerance factors: |y - y_ref| <= tau * sum_j |a_ij x_j|
TAU = {np.dtype(np.float64): 1e-12, np.dtype(np.float32): 1e-5}


def check_rows(y_test, ref: dict, dtype, exact: bool = False):
    """Apply the acceptance rule to a computed y against an oracle result.

    ``exact``: bitwise equality with the once-rounded oracle value (integer-valued
    inputs).  Otherwise |y - y_ref| <= tau * scale per row, with y_ref the long
    double result; a row whose scale is 0 must be exactly 0.
    Returns (ok, worst_ratio, index_of_worst).
    """
    dt = np.dtype(dtype)
    y_test = np.asarray(y_test)
    if exact:
        a = np.ascontiguousarray(y_test.astype(dt)).view(np.uint64 if dt == np.float64 else np.uint32)
        b = np.ascontiguousarray(ref["y"].astype(dt)).view(a.dtype)
        bad = np.nonzero(a != b)[0]
        return bad.size == 0, float(bad.size), int(bad[0]) if bad.size else -1
    yt = y_test.astype(np.float64)
    err = np.abs((yt - ref["y_hi"]) - ref["y_lo"])
    scale = ref["scale"]
    tol = TAU[dt] * scale
    finite = np.isfinite(yt)
    zero_scale = scale == 0
    ok_rows = finite & np.where(zero_scale, yt == 0, err <= tol)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(zero_scale, np.where(yt == 0, 0.0, np.inf), err / np.where(tol > 0, tol, 1))
    ratio = np.where(finite, ratio, np.inf)
    worst = int(np.argmax(ratio)) if ratio.size else -1
    return bool(ok_rows.all()), float(ratio[worst]) if ratio.size else 0.0, worst
