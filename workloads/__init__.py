"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This package only *builds* matrices and vectors; it holds no sparse matrix-vector
arithmetic.  See :mod:`workloads.generators`.
"""
from .generators import (  # noqa: F401
    CSR,
    laplacian_1d,
    laplacian_2d,
    laplacian_3d,
    laplacian_3d_relabelled,
    hmep_like,
    power_law,
    random_uniform_rows,
    banded_random_rows,
    convection_diffusion,
    random_csr,
    identity,
    permutation_matrix,
    uniform_x,
    integer_x,
    WORKLOADS,
    make_workload,
)
