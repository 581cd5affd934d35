"""BiCGSTAB for A x = b -- oracle, TEST INFRASTRUCTURE ONLY.

The Krylov/AMG paper solves its 3D Poisson test systems with BiCGSTAB (its Algorithm 4,
whose steps the extract does not carry).  This follows the textbook method of van der
Vorst (1992), unpreconditioned, with the shadow residual r_hat = r_0:

    rho_0 = alpha = omega = 1,  v_0 = p_0 = 0
    for k = 1, 2, ...
        rho_k = (r_hat, r_{k-1})
        beta  = (rho_k / rho_{k-1}) (alpha / omega)
        p_k   = r_{k-1} + beta (p_{k-1} - omega v_{k-1})
        v_k   = A p_k
        alpha = rho_k / (r_hat, v_k)
        s     = r_{k-1} - alpha v_k
        t     = A s
        omega = (t, s) / (t, t)          (0 when t = 0)
        x_k   = x_{k-1} + alpha p_k + omega s
        r_k   = s - omega t

Stopping rule (a reading, as for CG): stop before step k when ||r_{k-1}||_2 <= rtol ||b||_2
(||b|| -> 1 when b = 0), comparing squared norms in double, or after max_iter steps.
A zero rho_k or (r_hat, v_k) is a breakdown (ArithmeticError).

Arithmetic: float64 vectors and dot products (numpy); A p from :func:`oracle.spmv`
(long double, rounded to double); single-precision matrices are widened exactly.
Pinned by ``tests/test_bicgstab_oracle_pins.py``.  ``_mutation`` plants one mistake for
those pins (1: omega dropped from p; 2: wrong sign in s; 3: beta without alpha/omega).
"""
from __future__ import annotations

import numpy as np

from . import spmv


def bicgstab(csr, b, x0=None, rtol=1e-8, max_iter=1000, lib=None, _mutation=0) -> dict:
    A = csr if np.dtype(csr.vals.dtype) == np.float64 else csr.astype(np.float64)
    b = np.asarray(b, dtype=np.float64)
    x = np.zeros(A.n) if x0 is None else np.array(x0, dtype=np.float64)

    def matvec(u):
        return spmv(A, u, lib=lib)["y_hi"]

    r = b - matvec(x)
    r_hat = r.copy()
    bb = float(np.dot(b, b))
    denom = bb if bb > 0.0 else 1.0
    stop_rr = rtol * rtol * denom
    rr = float(np.dot(r, r))
    residuals = [np.sqrt(rr / denom)]
    rho_prev = alpha = omega = 1.0
    v = np.zeros(A.n)
    p = np.zeros(A.n)
    k = 0
    while k < max_iter and rr > stop_rr:
        rho = float(np.dot(r_hat, r))
        if rho == 0.0:
            raise ArithmeticError("BiCGSTAB breakdown: (r_hat, r) = 0")
        beta = (rho / rho_prev) if _mutation == 3 else (rho / rho_prev) * (alpha / omega)
        p = r + beta * (p - v) if _mutation == 1 else r + beta * (p - omega * v)
        v = matvec(p)
        rv = float(np.dot(r_hat, v))
        if rv == 0.0:
            raise ArithmeticError("BiCGSTAB breakdown: (r_hat, A p) = 0")
        alpha = rho / rv
        s = r + alpha * v if _mutation == 2 else r - alpha * v
        t = matvec(s)
        tt = float(np.dot(t, t))
        omega = float(np.dot(t, s)) / tt if tt > 0.0 else 0.0
        x = x + alpha * p + omega * s
        r = s - omega * t
        rr = float(np.dot(r, r))
        rho_prev = rho
        k += 1
        residuals.append(np.sqrt(rr / denom))
        if omega == 0.0 and rr > stop_rr:
            raise ArithmeticError("BiCGSTAB breakdown: omega = 0")
    return {"x": x, "iterations": k, "residuals": np.array(residuals)}
