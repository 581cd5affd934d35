"""Restarted GMRES(m) for A x = b -- oracle, TEST INFRASTRUCTURE ONLY.

The Krylov/AMG paper names GMRES among the Krylov solvers it implements (solvers
section, beside CG and BiCGSTAB) but prints none of its steps.  This follows the
generalized minimal residual method of Saad and Schultz (1986), unpreconditioned:

    r = b - A x, beta = ||r||
    cycle:  v_0 = r / beta, g = beta e_1
        for j = 0 .. m-1:
            w = A v_j
            h = V^T w, w -= V h, c = V^T w, w -= V c, h += c      (V = [v_0 .. v_j];
                                                                   Gram-Schmidt twice)
            h_{j+1} = ||w||
            apply the rotations G_0 .. G_{j-1} to (h_0 .. h_j), then the rotation G_j
            that zeroes h_{j+1}: (c_j, s_j) = (h_j, h_{j+1}) / hypot(h_j, h_{j+1});
            g_{j+1} = -s_j g_j, g_j = c_j g_j
            one step done; stop the cycle when |g_{j+1}| <= rtol ||b||, when h_{j+1} = 0
            (the Krylov space is invariant: the cycle's solution is exact) or at max_iter
            v_{j+1} = w / h_{j+1}
        solve the upper triangular R y = g_{0..j}; x += V y
        r = b - A x, beta = ||r||; stop when beta <= rtol ||b|| or at max_iter

Readings (the pages give none of this): ||b|| is replaced by 1 when b = 0; the
iteration count is the number of Arnoldi steps over all cycles; the final relative
residual is the true one, ||b - A x|| / ||b||.

Arithmetic: float64 vectors and dot products (numpy); A v from :func:`oracle.spmv`
(long double, rounded to double).  Pinned by ``tests/test_gmres_oracle_pins.py``.
``_mutation`` plants one mistake for those pins (1: wrong sign of s in the rotation;
2: the back-substitution leaves the last unknown at 0; 3: g not rotated).  A zero
pivot of R (A singular on the Krylov space) is a breakdown (ArithmeticError).
"""
from __future__ import annotations

import numpy as np

from . import spmv


def gmres(csr, b, x0=None, m=30, rtol=1e-8, max_iter=1000, lib=None, _mutation=0) -> dict:
    A = csr if np.dtype(csr.vals.dtype) == np.float64 else csr.astype(np.float64)
    b = np.asarray(b, dtype=np.float64)
    n = A.n
    x = np.zeros(n) if x0 is None else np.array(x0, dtype=np.float64)

    def matvec(u):
        return spmv(A, u, lib=lib)["y_hi"]

    bnorm = float(np.sqrt(np.dot(b, b)))
    denom = bnorm if bnorm > 0.0 else 1.0
    tol = rtol * denom
    r = b - matvec(x)
    beta = float(np.sqrt(np.dot(r, r)))
    residuals = [beta / denom]  # true residual at the start of every cycle, and at the end
    estimates = []              # |g_{j+1}| / ||b|| after every Arnoldi step
    k = 0
    while beta > tol and k < max_iter:
        V = np.zeros((m + 1, n))
        H = np.zeros((m + 1, m))
        cs = np.zeros(m)
        sn = np.zeros(m)
        g = np.zeros(m + 1)
        V[0] = r / beta
        g[0] = beta
        steps = 0
        for j in range(m):
            w = matvec(V[j])
            h = V[: j + 1] @ w
            w = w - V[: j + 1].T @ h
            c = V[: j + 1] @ w
            w = w - V[: j + 1].T @ c
            h = h + c
            hn = float(np.sqrt(np.dot(w, w)))
            col = np.concatenate([h, [hn]])
            for i in range(j):  # the earlier rotations
                a, bb = col[i], col[i + 1]
                col[i] = cs[i] * a + sn[i] * bb
                col[i + 1] = -sn[i] * a + cs[i] * bb
            rho = float(np.hypot(col[j], col[j + 1]))
            cs[j] = col[j] / rho if rho > 0.0 else 1.0
            sn[j] = col[j + 1] / rho if rho > 0.0 else 0.0
            if _mutation == 1:
                sn[j] = -sn[j]
            col[j] = cs[j] * col[j] + sn[j] * col[j + 1]
            col[j + 1] = 0.0
            H[: j + 2, j] = col
            if _mutation != 3:
                g[j + 1] = -sn[j] * g[j]
                g[j] = cs[j] * g[j]
            steps = j + 1
            k += 1
            estimates.append(abs(g[j + 1]) / denom)
            if abs(g[j + 1]) <= tol or hn == 0.0 or k >= max_iter:
                break
            V[j + 1] = w / hn
        # back-substitution R y = g
        y = np.zeros(steps)
        last = steps - 1 if _mutation == 2 else steps
        for i in range(last - 1, -1, -1):
            if H[i, i] == 0.0:
                raise ArithmeticError("GMRES breakdown: zero pivot in the rotated Hessenberg matrix")
            y[i] = (g[i] - H[i, i + 1:steps] @ y[i + 1:steps]) / H[i, i]
        x = x + V[:steps].T @ y
        r = b - matvec(x)
        beta = float(np.sqrt(np.dot(r, r)))
        residuals.append(beta / denom)
    return {"x": x, "iterations": k, "residuals": np.array(residuals), "estimates": np.array(estimates),
            "relative_residual": beta / denom}
