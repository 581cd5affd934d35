"""Closed forms for conjugate gradients on Dirichlet Laplacians (no solver code here).

The eigenvalues of the Dirichlet Laplacian on an n_1 x ... x n_d grid (diagonal 2d,
neighbours -1) are sums over the axes of 2 - 2 cos(k pi / (n + 1)), k = 1..n.  The
textbook CG bound ||e_k||_A <= 2 rho^k ||e_0||_A with rho = (sqrt(kappa) - 1) /
(sqrt(kappa) + 1) gives, for the 2-norm residual from x_0 = 0,
||r_k|| <= 2 sqrt(kappa) rho^k ||b||.
"""
import math


def laplacian_extreme_eigenvalues(dims):
    lo = sum(2.0 - 2.0 * math.cos(math.pi / (n + 1)) for n in dims)
    hi = sum(2.0 + 2.0 * math.cos(math.pi / (n + 1)) for n in dims)
    return lo, hi


def cg_iteration_bound(dims, rtol):
    """Smallest k for which the bound guarantees ||r_k|| <= rtol ||b|| (x_0 = 0)."""
    lo, hi = laplacian_extreme_eigenvalues(dims)
    sk = math.sqrt(hi / lo)
    rho = (sk - 1.0) / (sk + 1.0)
    return max(0, math.ceil(math.log(rtol / (2.0 * sk)) / math.log(rho)))
