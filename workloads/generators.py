"""Seeded synthetic sparse matrices and vectors.

Every matrix is returned in CSR form (``row_ptr`` int32 [n+1], ``col_idx`` int32
[nnz], ``vals`` float64/float32 [nnz]) with columns sorted and free of duplicates
inside each row (fill-complete, as the Trilinos issue "Tpetra::CrsMatrix::
unpackAndCombine: Optimize GPU unpack for few long rows" assumes of a finished
matrix), unless a generator is asked for duplicates or unsorted rows on purpose.

The shapes stand in for the matrices the pages measure on, none of which is
available here:

* 2D / 3D Laplacian stencils (Dirichlet, natural ordering) stand in for the
  3D_Poisson matrices of "Development of Krylov and AMG linear solvers for
  large-scale sparse matrices on GPUs" (numerical experiments section).
* :func:`hmep_like` copies the shape the GPGPU spMVM paper (arXiv 1112.5588,
  test-matrix section) gives for HMEp: dimension 6.2e6, about 15 non-zeros per
  row, off-diagonals made of unbroken runs 15,000 entries long.
* :func:`power_law` is an irregular matrix with a few nearly dense rows, the case
  "Load-balancing Sparse Matrix Vector Product Kernels on GPUs" (abstract) and the
  Trilinos issue (description) single out.
* :func:`random_uniform_rows` has constant row length and no x locality.

This module builds inputs only; it contains no matrix-vector arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# --------------------------------------------------------------------------- #
# container
# --------------------------------------------------------------------------- #


@dataclass
class CSR:
    """A square n x n matrix in compressed sparse row form."""

    n: int
    row_ptr: np.ndarray
    col_idx: np.ndarray
    vals: np.ndarray
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1])

    @property
    def dtype(self):
        return self.vals.dtype

    def row_lengths(self) -> np.ndarray:
        return np.diff(self.row_ptr.astype(np.int64))

    def astype(self, dtype) -> "CSR":
        return CSR(self.n, self.row_ptr, self.col_idx, self.vals.astype(dtype), self.name, dict(self.meta))


def _check_index_range(n: int, nnz: int) -> None:
    if n >= 2**31 or nnz >= 2**31:
        raise ValueError("n and nnz must stay below 2^31 for int32 indices")


def _csr_from_mask(n, cols, mask, vals_full, dtype, name, meta=None) -> CSR:
    """Keep the masked candidate entries of an (n, k) candidate table, row-major."""
    lens = mask.sum(axis=1, dtype=np.int64)
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(lens, out=row_ptr[1:])
    _check_index_range(n, int(row_ptr[-1]))
    col_idx = cols[mask].astype(np.int32)
    vals = np.asarray(vals_full[mask], dtype=dtype)
    return CSR(n, row_ptr.astype(np.int32), col_idx, vals, name, meta or {})


# --------------------------------------------------------------------------- #
# stencils
# --------------------------------------------------------------------------- #


def laplacian_1d(n: int, dtype=np.float64) -> CSR:
    """tridiag(-1, 2, -1), Dirichlet ends."""
    idx = np.arange(n, dtype=np.int64)
    offs = np.array([-1, 0, 1], dtype=np.int64)
    cols = idx[:, None] + offs[None, :]
    mask = (cols >= 0) & (cols < n)
    vals = np.broadcast_to(np.array([-1.0, 2.0, -1.0])[None, :], cols.shape)
    return _csr_from_mask(n, cols, mask, vals, dtype, f"lap1d_{n}")


def laplacian_2d(nx: int, ny: int, dtype=np.float64) -> CSR:
    """5-point Dirichlet Laplacian on an nx x ny grid: diagonal 4, neighbours -1.

    Row r = i + nx*j (natural ordering); columns sorted ascending.
    """
    n = nx * ny
    idx = np.arange(n, dtype=np.int64)
    i = idx % nx
    j = idx // nx
    offs = np.array([-nx, -1, 0, 1, nx], dtype=np.int64)
    cols = idx[:, None] + offs[None, :]
    mask = np.stack([j > 0, i > 0, np.ones(n, bool), i < nx - 1, j < ny - 1], axis=1)
    vals = np.broadcast_to(np.array([-1.0, -1.0, 4.0, -1.0, -1.0])[None, :], cols.shape)
    return _csr_from_mask(n, cols, mask, vals, dtype, f"lap2d_{nx}x{ny}", {"grid": (nx, ny)})


def laplacian_3d(nx: int, ny: int, nz: int, dtype=np.float64) -> CSR:
    """7-point Dirichlet Laplacian on an nx x ny x nz grid: diagonal 6, neighbours -1.

    Row r = i + nx*(j + ny*k) (natural ordering); columns sorted ascending.
    """
    n = nx * ny * nz
    idx = np.arange(n, dtype=np.int64)
    i = idx % nx
    j = (idx // nx) % ny
    k = idx // (nx * ny)
    offs = np.array([-nx * ny, -nx, -1, 0, 1, nx, nx * ny], dtype=np.int64)
    cols = idx[:, None] + offs[None, :]
    mask = np.stack(
        [k > 0, j > 0, i > 0, np.ones(n, bool), i < nx - 1, j < ny - 1, k < nz - 1], axis=1
    )
    vals = np.broadcast_to(np.array([-1.0, -1.0, -1.0, 6.0, -1.0, -1.0, -1.0])[None, :], cols.shape)
    return _csr_from_mask(n, cols, mask, vals, dtype, f"lap3d_{nx}x{ny}x{nz}", {"grid": (nx, ny, nz)})


def laplacian_3d_relabelled(nx: int, ny: int, nz: int, seed: int = 9, dtype=np.float64) -> CSR:
    """The 7-point Dirichlet Laplacian with its grid points numbered in a seeded random
    order: grid point p gets the label lab[p] (a random bijection), its row is lab[p],
    and its neighbours q appear as columns lab[q].  Columns sorted ascending.  The same
    operator as ``laplacian_3d`` with its locality destroyed: the input for which a
    bandwidth-reducing ordering matters."""
    n = nx * ny * nz
    lab = np.random.default_rng(seed).permutation(n).astype(np.int64)
    idx = np.arange(n, dtype=np.int64)
    i = idx % nx
    j = (idx // nx) % ny
    k = idx // (nx * ny)
    offs = np.array([-nx * ny, -nx, -1, 0, 1, nx, nx * ny], dtype=np.int64)
    nb = idx[:, None] + offs[None, :]
    mask = np.stack([k > 0, j > 0, i > 0, np.ones(n, bool), i < nx - 1, j < ny - 1, k < nz - 1], axis=1)
    val_row = np.array([-1.0, -1.0, -1.0, 6.0, -1.0, -1.0, -1.0])
    rows = np.broadcast_to(lab[:, None], nb.shape)[mask]
    cols = lab[np.where(mask, nb, 0)][mask]
    vals = np.broadcast_to(val_row[None, :], nb.shape)[mask]
    order = np.lexsort((cols, rows))
    rows, cols, vals = rows[order], cols[order], vals[order]
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.add.at(row_ptr, rows + 1, 1)
    row_ptr = np.cumsum(row_ptr)
    _check_index_range(n, int(row_ptr[-1]))
    return CSR(n, row_ptr.astype(np.int32), cols.astype(np.int32), vals.astype(dtype),
               f"lap3d_{nx}x{ny}x{nz}_relabelled", {"grid": (nx, ny, nz), "labels": lab})


def convection_diffusion(dims, c: float = 0.5, dtype=np.float64) -> CSR:
    """Upwind convection-diffusion on a Dirichlet grid (1 to 3 dimensions), flow along the
    first axis: the Laplacian stencil (diagonal 2d, neighbours -1) plus c on the diagonal
    and -c on the upstream neighbour.  Nonsymmetric, diagonally dominant (an M-matrix).
    Row r = i0 + n0 (i1 + n1 i2); columns sorted ascending."""
    dims = tuple(int(d) for d in dims)
    n = int(np.prod(dims))
    idx = np.arange(n, dtype=np.int64)
    coord, rest = [], idx
    for d in dims:
        coord.append(rest % d)
        rest = rest // d
    strides = np.cumprod((1,) + dims[:-1])
    offs, masks, vals = [], [], []
    for a in reversed(range(len(dims))):
        offs.append(-strides[a]); masks.append(coord[a] > 0); vals.append(-1.0 - (c if a == 0 else 0.0))
    offs.append(0); masks.append(np.ones(n, bool)); vals.append(2.0 * len(dims) + c)
    for a in range(len(dims)):
        offs.append(strides[a]); masks.append(coord[a] < dims[a] - 1); vals.append(-1.0)
    cols = idx[:, None] + np.array(offs, dtype=np.int64)[None, :]
    mask = np.stack(masks, axis=1)
    vfull = np.broadcast_to(np.array(vals)[None, :], cols.shape)
    return _csr_from_mask(n, cols, mask, vfull, dtype, "convdiff_" + "x".join(map(str, dims)), {"grid": dims, "c": c})


# --------------------------------------------------------------------------- #
# HMEp-shaped
# --------------------------------------------------------------------------- #

#: positive half of the off-diagonal offset set (22 offsets with the negatives)
HMEP_OFFSETS = (1, 6, 36, 216, 1296, 15000, 30000, 90000, 180000, 540000, 1080000)


def hmep_like(
    n: int = 6_200_000,
    block: int = 15_000,
    seed: int = 3,
    p_include: float = 14.0 / 22.0,
    min_offdiag: int = 7,
    max_offdiag: int = 21,
    offsets=HMEP_OFFSETS,
    dtype=np.float64,
    chunk: int = 1 << 20,
) -> CSR:
    """Holstein-Hubbard-shaped synthetic matrix.

    For every block of ``block`` consecutive rows each of the 22 off-diagonal
    offsets (+-``offsets``) is switched on with probability ``p_include``; a block
    is redrawn until it has between ``min_offdiag`` and ``max_offdiag`` offsets.
    Each row holds its diagonal plus the switched-on offsets that stay inside the
    matrix, so interior rows have 8..22 entries (mean about 15) and every
    switched-on offset forms a contiguous off-diagonal run ``block`` rows long.
    Off-diagonal values are N(0, 1), diagonal values N(0, 4) (standard deviation 2).
    """
    rng = np.random.default_rng(seed)
    offs = np.array(sorted([-o for o in offsets] + list(offsets)), dtype=np.int64)
    n_off = offs.size
    nblocks = -(-n // block)
    incl = rng.random((nblocks, n_off)) < p_include
    while True:
        cnt = incl.sum(axis=1)
        bad = np.nonzero((cnt < min_offdiag) | (cnt > max_offdiag))[0]
        if bad.size == 0:
            break
        incl[bad] = rng.random((bad.size, n_off)) < p_include
    all_offs = np.concatenate([offs[offs < 0], [0], offs[offs > 0]])
    diag_col = int(np.nonzero(all_offs == 0)[0][0])
    incl_all = np.concatenate(
        [incl[:, :diag_col], np.ones((nblocks, 1), bool), incl[:, diag_col:]], axis=1)
    lens = np.empty(n, dtype=np.int64)
    cols_parts, diag_parts = [], []
    for r0 in range(0, n, chunk):
        r1 = min(n, r0 + chunk)
        rows = np.arange(r0, r1, dtype=np.int64)
        cand = rows[:, None] + all_offs[None, :]
        mask = incl_all[rows // block] & (cand >= 0) & (cand < n)
        lens[r0:r1] = mask.sum(axis=1)
        cols_parts.append(cand[mask].astype(np.int32))
        isd = np.zeros(mask.shape, bool)
        isd[:, diag_col] = True
        diag_parts.append(isd[mask])
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(lens, out=row_ptr[1:])
    _check_index_range(n, int(row_ptr[-1]))
    col_idx = np.concatenate(cols_parts)
    is_diag = np.concatenate(diag_parts)
    vals = rng.standard_normal(col_idx.size)
    vals[is_diag] *= 2.0
    return CSR(n, row_ptr.astype(np.int32), col_idx, vals.astype(dtype), f"hmep_like_{n}",
               {"block": block, "offsets": offs.tolist()})


# --------------------------------------------------------------------------- #
# power law
# --------------------------------------------------------------------------- #


def _sorted_distinct_rows(rng, n, row_ptr, lens, dense_rows):
    """Column indices, uniform over [0, n), distinct and sorted inside each row."""
    nnz = int(row_ptr[-1])
    cols = rng.integers(0, n, size=nnz, dtype=np.int64)
    for r in dense_rows:
        a, b = int(row_ptr[r]), int(row_ptr[r + 1])
        cols[a:b] = rng.choice(n, size=b - a, replace=False)
    row_of = np.repeat(np.arange(n, dtype=np.int64), lens)
    key = row_of * n + cols
    key.sort()
    dense_set = np.zeros(n, bool)
    dense_set[np.asarray(dense_rows, dtype=np.int64)] = True
    # Fix duplicates only inside the rows that have some; draws w/o replacement never do.
    while True:
        dup = np.nonzero(key[1:] == key[:-1])[0] + 1
        if dup.size == 0:
            break
        bad_rows = np.unique(key[dup] // n)
        assert not dense_set[bad_rows].any()
        for r in bad_rows:
            a, b = int(row_ptr[r]), int(row_ptr[r + 1])
            seg = np.unique(key[a:b] - r * n)
            while seg.size < b - a:
                extra = rng.integers(0, n, size=(b - a) - seg.size, dtype=np.int64)
                seg = np.unique(np.concatenate([seg, extra]))
            key[a:b] = seg + r * n
    return (key - row_of * n).astype(np.int32)


def power_law(
    n: int = 4_000_000,
    zipf_s: float = 2.0,
    zipf_max: int = 100_000,
    n_dense: int = 32,
    dense_lo: int = 200_000,
    dense_hi: int = 1_000_000,
    seed: int = 4,
    dtype=np.float64,
) -> CSR:
    """Irregular matrix: Zipf row lengths plus a few nearly dense rows.

    Row lengths follow a Zipf law with exponent ``zipf_s`` truncated to
    [1, ``zipf_max``]; ``n_dense`` rows at seeded random positions get lengths
    uniform on [``dense_lo``, ``dense_hi``].  Columns are uniform over [0, n),
    distinct and sorted inside each row; values are N(0, 1).
    """
    rng = np.random.default_rng(seed)
    k = np.arange(1, min(zipf_max, n) + 1, dtype=np.float64)
    pmf = k ** (-zipf_s)
    cdf = np.cumsum(pmf)
    cdf /= cdf[-1]
    lens = np.searchsorted(cdf, rng.random(n), side="right").astype(np.int64) + 1
    lens = np.minimum(lens, min(zipf_max, n))
    dense_rows = np.sort(rng.choice(n, size=min(n_dense, n), replace=False))
    dense_lens = rng.integers(min(dense_lo, n), min(dense_hi, n) + 1, size=dense_rows.size)
    lens[dense_rows] = dense_lens
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(lens, out=row_ptr[1:])
    _check_index_range(n, int(row_ptr[-1]))
    cols = _sorted_distinct_rows(rng, n, row_ptr, lens, dense_rows)
    vals = rng.standard_normal(cols.size).astype(dtype)
    return CSR(n, row_ptr.astype(np.int32), cols, vals, f"power_law_{n}",
               {"dense_rows": dense_rows.tolist()})


# --------------------------------------------------------------------------- #
# random uniform
# --------------------------------------------------------------------------- #


def random_uniform_rows(n: int = 16_777_216, per_row: int = 16, seed: int = 5, dtype=np.float32) -> CSR:
    """Exactly ``per_row`` distinct, sorted, uniformly random columns per row; values U(-1, 1)."""
    rng = np.random.default_rng(seed)
    per_row = min(per_row, n)
    cols = rng.integers(0, n, size=(n, per_row), dtype=np.int32)
    cols.sort(axis=1)
    bad = np.nonzero((cols[:, 1:] == cols[:, :-1]).any(axis=1))[0]
    while bad.size:
        redo = rng.integers(0, n, size=(bad.size, per_row), dtype=np.int32)
        redo.sort(axis=1)
        cols[bad] = redo
        still = (redo[:, 1:] == redo[:, :-1]).any(axis=1)
        bad = bad[still]
    nnz = n * per_row
    _check_index_range(n, nnz)
    row_ptr = (np.arange(n + 1, dtype=np.int64) * per_row).astype(np.int32)
    if np.dtype(dtype) == np.float32:
        vals = rng.random(nnz, dtype=np.float32) * np.float32(2) - np.float32(1)
    else:
        vals = (rng.random(nnz) * 2.0 - 1.0).astype(dtype)
    return CSR(n, row_ptr, cols.reshape(-1), vals, f"uniform{per_row}_{n}")


def banded_random_rows(n: int, per_row: int, half_band: int, seed: int = 6, dtype=np.float64) -> CSR:
    """Exactly ``per_row`` distinct, sorted columns per row, uniform in the band
    [i - half_band, i + half_band] clipped to [0, n); values U(-1, 1).  Wide rows with a
    local x footprint: the shape for which several threads share a row."""
    rng = np.random.default_rng(seed)
    rows = np.arange(n, dtype=np.int64)
    lo = np.maximum(rows - half_band, 0)
    hi = np.minimum(rows + half_band, n - 1)
    per_row = int(min(per_row, int((hi - lo + 1).min())))
    span = (hi - lo + 1)[:, None]
    cols = lo[:, None] + (rng.random((n, per_row)) * span).astype(np.int64)
    cols.sort(axis=1)
    bad = np.nonzero((cols[:, 1:] == cols[:, :-1]).any(axis=1))[0]
    while bad.size:
        redo = lo[bad, None] + (rng.random((bad.size, per_row)) * span[bad]).astype(np.int64)
        redo.sort(axis=1)
        cols[bad] = redo
        bad = bad[(redo[:, 1:] == redo[:, :-1]).any(axis=1)]
    nnz = n * per_row
    _check_index_range(n, nnz)
    row_ptr = (np.arange(n + 1, dtype=np.int64) * per_row).astype(np.int32)
    vals = (rng.random(nnz) * 2.0 - 1.0).astype(dtype)
    return CSR(n, row_ptr, cols.reshape(-1).astype(np.int32), vals, f"band{per_row}_{n}")


# --------------------------------------------------------------------------- #
# tiny matrices for pins
# --------------------------------------------------------------------------- #


def random_csr(
    n: int,
    density: float,
    seed: int,
    dtype=np.float64,
    integer_values: bool = False,
    duplicates: bool = False,
    unsorted: bool = False,
    empty_row_fraction: float = 0.0,
    full_rows: int = 0,
) -> CSR:
    """Small random square CSR with optional duplicates, unsorted rows, empty and full rows."""
    rng = np.random.default_rng(seed)
    rows = []
    full = set(rng.choice(n, size=min(full_rows, n), replace=False).tolist()) if full_rows else set()
    for r in range(n):
        if r in full:
            c = np.arange(n)
        elif rng.random() < empty_row_fraction:
            c = np.zeros(0, dtype=np.int64)
        else:
            m = rng.binomial(n, density)
            if duplicates:
                c = np.sort(rng.integers(0, n, size=m))
            else:
                c = np.sort(rng.choice(n, size=m, replace=False))
        if unsorted:
            c = rng.permutation(c)
        rows.append(np.asarray(c, dtype=np.int64))
    lens = np.array([len(c) for c in rows], dtype=np.int64)
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(lens, out=row_ptr[1:])
    col_idx = np.concatenate(rows).astype(np.int32) if rows else np.zeros(0, np.int32)
    if integer_values:
        vals = rng.integers(-8, 9, size=col_idx.size).astype(dtype)
    else:
        vals = rng.standard_normal(col_idx.size).astype(dtype)
    return CSR(n, row_ptr.astype(np.int32), col_idx, vals, f"random_{n}_{density}")


def identity(n: int, dtype=np.float64) -> CSR:
    return CSR(n, np.arange(n + 1, dtype=np.int32), np.arange(n, dtype=np.int32),
               np.ones(n, dtype=dtype), f"identity_{n}")


def permutation_matrix(perm, dtype=np.float64) -> CSR:
    """Row i holds a single 1 at column perm[i], so (P x)_i = x[perm[i]]."""
    perm = np.asarray(perm, dtype=np.int32)
    n = perm.size
    return CSR(n, np.arange(n + 1, dtype=np.int32), perm.copy(), np.ones(n, dtype=dtype), f"perm_{n}")


# --------------------------------------------------------------------------- #
# vectors
# --------------------------------------------------------------------------- #


def uniform_x(n: int, seed: int = 101, dtype=np.float64) -> np.ndarray:
    """x uniform on [-1, 1)."""
    rng = np.random.default_rng(seed)
    if np.dtype(dtype) == np.float32:
        return rng.random(n, dtype=np.float32) * np.float32(2) - np.float32(1)
    return (rng.random(n) * 2.0 - 1.0).astype(dtype)


def integer_x(n: int, lo: int = -8, hi: int = 8, seed: int = 102, dtype=np.float64) -> np.ndarray:
    """Integer-valued x uniform on {lo, ..., hi}."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=n).astype(dtype)


# --------------------------------------------------------------------------- #
# named workloads
# --------------------------------------------------------------------------- #

WORKLOADS = {
    # full-size workloads
    "lap2d_256": dict(fn=laplacian_2d, kw=dict(nx=256, ny=256), dtype=np.float64, seed_x=101,
                      desc="2D 5-point Laplacian 256x256, Dirichlet, n=65,536"),
    "lap3d_128": dict(fn=laplacian_3d, kw=dict(nx=128, ny=128, nz=128), dtype=np.float64, seed_x=101,
                      desc="3D 7-point Laplacian 128^3, Dirichlet, n=2,097,152"),
    "hmep_6p2m": dict(fn=hmep_like, kw=dict(n=6_200_000, seed=3), dtype=np.float64, seed_x=101,
                      desc="HMEp-shaped synthetic, n=6,200,000, ~15 nnz/row"),
    "powerlaw_4m": dict(fn=power_law, kw=dict(n=4_000_000, seed=4), dtype=np.float64, seed_x=101,
                        desc="power-law Zipf(2) rows + 32 dense rows of 200k-1M, n=4,000,000"),
    "uniform16_16m": dict(fn=random_uniform_rows, kw=dict(n=16_777_216, per_row=16, seed=5),
                          dtype=np.float32, seed_x=101,
                          desc="random uniform, 16 nnz/row, n=16,777,216"),
    # wide rows, few of them: the regime of several threads per row
    "lap3d_128_relabelled": dict(fn=laplacian_3d_relabelled, kw=dict(nx=128, ny=128, nz=128, seed=9),
                                 dtype=np.float64, seed_x=101,
                                 desc="3D 7-point Laplacian 128^3 with randomly numbered grid points"),
    "convdiff3d_128": dict(fn=convection_diffusion, kw=dict(dims=(128, 128, 128), c=0.5), dtype=np.float64,
                           seed_x=101, desc="3D upwind convection-diffusion 128^3 (nonsymmetric), n=2,097,152"),
    "band120_256k": dict(fn=banded_random_rows, kw=dict(n=262_144, per_row=120, half_band=4096, seed=6),
                         dtype=np.float64, seed_x=101,
                         desc="banded random, 120 nnz/row in a band of +-4096, n=262,144"),
    "band128_32k": dict(fn=banded_random_rows, kw=dict(n=32_768, per_row=128, half_band=2048, seed=7),
                        dtype=np.float64, seed_x=101,
                        desc="banded random, 128 nnz/row in a band of +-2048, n=32,768"),
    # small versions of the same shapes (several tiles and a ragged tail)
    "lap2d_small": dict(fn=laplacian_2d, kw=dict(nx=67, ny=45), dtype=np.float64, seed_x=101,
                        desc="2D 5-point Laplacian 67x45"),
    "lap3d_small": dict(fn=laplacian_3d, kw=dict(nx=37, ny=29, nz=23), dtype=np.float64, seed_x=101,
                        desc="3D 7-point Laplacian 37x29x23"),
    "hmep_small": dict(fn=hmep_like, kw=dict(n=160_003, block=15_000, seed=3), dtype=np.float64,
                       seed_x=101, desc="HMEp-shaped, n=160,003"),
    "powerlaw_small": dict(fn=power_law, kw=dict(n=60_001, zipf_max=3000, n_dense=4, dense_lo=9000,
                                                 dense_hi=40000, seed=4),
                           dtype=np.float64, seed_x=101, desc="power law, n=60,001 with 4 dense rows"),
    "lap3d_relabelled_small": dict(fn=laplacian_3d_relabelled, kw=dict(nx=37, ny=29, nz=23, seed=9),
                                   dtype=np.float64, seed_x=101, desc="3D Laplacian 37x29x23, random numbering"),
    "convdiff_small": dict(fn=convection_diffusion, kw=dict(dims=(41, 33, 19), c=0.5), dtype=np.float64,
                           seed_x=101, desc="3D convection-diffusion 41x33x19"),
    "band_small": dict(fn=banded_random_rows, kw=dict(n=20_011, per_row=96, half_band=700, seed=8),
                       dtype=np.float64, seed_x=101, desc="banded random 96/row, n=20,011"),
    "uniform16_small": dict(fn=random_uniform_rows, kw=dict(n=100_003, per_row=16, seed=5),
                            dtype=np.float32, seed_x=101, desc="random uniform 16/row, n=100,003"),
}


def make_workload(name: str, dtype=None, integer_x_values: bool = False):
    """Return (CSR, x) for a named workload; ``dtype`` overrides the value type."""
    spec = WORKLOADS[name]
    dt = np.dtype(dtype if dtype is not None else spec["dtype"])
    kw = dict(spec["kw"])
    csr = spec["fn"](dtype=dt, **kw)
    if integer_x_values:
        x = integer_x(csr.n, dtype=dt)
    else:
        x = uniform_x(csr.n, seed=spec["seed_x"], dtype=dt)
    csr.name = name
    return csr, x
