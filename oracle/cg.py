"""Conjugate gradients for A x = b -- oracle, TEST INFRASTRUCTURE ONLY.

The Krylov/AMG paper lists CG among the Krylov subspace solvers it builds on its SpMV
and vector operations (section on Krylov subspace algorithms) but prints the steps of
BiCGSTAB only, pointing to the literature for the others.  This file therefore follows
the textbook method of Hestenes and Stiefel (1952), in its usual notation:

    r_0 = b - A x_0,   p_0 = r_0
    alpha_k = (r_k . r_k) / (p_k . A p_k)
    x_{k+1} = x_k + alpha_k p_k
    r_{k+1} = r_k - alpha_k A p_k
    beta_k  = (r_{k+1} . r_{k+1}) / (r_k . r_k)
    p_{k+1} = r_{k+1} + beta_k p_k

Stopping rule (a reading: the pages give none): stop before step k when
||r_k||_2 <= rtol * ||b||_2 (||b|| replaced by 1 when b = 0), comparing the squared
norms in double, or after max_iter steps.

Arithmetic: float64 vectors and dot products (numpy); A p from :func:`oracle.spmv`
(long double, rounded to double).  Single-precision matrices are widened exactly to
float64 first.  Pinned by ``tests/test_cg_oracle_pins.py`` against a dense solve, the
one-step eigenvector case, the distinct-eigenvalue count, the energy-norm decrease
and the Chebyshev convergence bound.

``_mutation`` plants one mistake for the pin tests (0: none; 1: beta divided by
p.Ap; 2: residual updated with the wrong sign; 3: the previous direction dropped
from p).
"""
from __future__ import annotations

import numpy as np

from . import spmv


def cg(csr, b, x0=None, rtol=1e-8, max_iter=1000, lib=None, _mutation=0) -> dict:
    """Run CG from ``x0`` (zeros when None).

    Returns ``x`` (float64), ``iterations`` and ``residuals`` (||r_k|| / ||b|| for
    k = 0 .. iterations, from the recurrence).
    """
    A = csr if np.dtype(csr.vals.dtype) == np.float64 else csr.astype(np.float64)
    b = np.asarray(b, dtype=np.float64)
    x = np.zeros(A.n) if x0 is None else np.array(x0, dtype=np.float64)

    def matvec(v):
        return spmv(A, v, lib=lib)["y_hi"]

    r = b - matvec(x)
    p = r.copy()
    rr = float(np.dot(r, r))
    bb = float(np.dot(b, b))
    denom = bb if bb > 0.0 else 1.0
    stop_rr = rtol * rtol * denom
    residuals = [np.sqrt(rr / denom)]
    k = 0
    while k < max_iter and rr > stop_rr:
        q = matvec(p)
        pq = float(np.dot(p, q))
        if not pq > 0.0:
            raise ArithmeticError("p.Ap <= 0: the matrix is not positive definite")
        alpha = rr / pq
        x = x + alpha * p
        r = r + alpha * q if _mutation == 2 else r - alpha * q
        rr_next = float(np.dot(r, r))
        beta = rr_next / (pq if _mutation == 1 else rr)
        p = r.copy() if _mutation == 3 else r + beta * p
        rr = rr_next
        k += 1
        residuals.append(np.sqrt(rr / denom))
    return {"x": x, "iterations": k, "residuals": np.array(residuals)}
