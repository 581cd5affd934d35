"""Storage-layout definitions the GPU formats must reproduce exactly.

TEST INFRASTRUCTURE ONLY (see the package docstring).

All functions take the row-length array ``lens`` (len_i = row_ptr[i+1] - row_ptr[i])
and return plain integers / arrays, so the GPU builder's integer work (row order,
slice widths, padded sizes, the ELL/COO split) can be compared bit for bit.

Sources
-------
* ELLPACK / ELLPACK-R: rows shifted left and stored as an N x N_nzr^max rectangle,
  with a row-length array so threads stop at their own row's end -- GPGPU spMVM
  paper (arXiv 1112.5588), ELLPACK-R section, Figs. 1-2.
* pJDS: rows sorted by length, longest first, then every block of b_r consecutive
  rows padded to the longest row in the block -- same paper, pJDS section, Fig. 1.
  SELL-C-sigma generalises the sort to windows of sigma rows (sigma = n is pJDS,
  sigma = 1 keeps the natural order) with slices of C = b_r rows.
* HYB / HEC: the first K entries of every row in an ELL part whose leading
  dimension is a multiple of 32 (256 in the Krylov/AMG paper), the rest of the row
  in a COO or CSR spill -- "Development of Krylov and AMG linear solvers ...",
  matrix-format section, Figs. 1-3.
"""
from __future__ import annotations

import numpy as np


def row_lengths(row_ptr) -> np.ndarray:
    rp = np.asarray(row_ptr, dtype=np.int64)
    return rp[1:] - rp[:-1]


def long_rows(lens, threshold: int) -> np.ndarray:
    """Rows longer than ``threshold`` (they leave the sliced part for the long-row pass)."""
    lens = np.asarray(lens, dtype=np.int64)
    return np.nonzero(lens > threshold)[0].astype(np.int64)


def sell_order(lens, sigma: int) -> np.ndarray:
    """Row order of SELL-C-sigma: inside each window of ``sigma`` consecutive rows,
    rows sorted by length, longest first; equal lengths keep their original order.

    Returns perm with perm[p] = original row stored at sorted position p.
    """
    lens = np.asarray(lens, dtype=np.int64)
    n = lens.size
    sigma = max(1, min(int(sigma), max(n, 1)))
    perm = np.empty(n, dtype=np.int64)
    for w0 in range(0, n, sigma):
        w1 = min(n, w0 + sigma)
        # stable sort on -length: longest first, ties keep the original order
        perm[w0:w1] = np.argsort(-lens[w0:w1], kind="stable") + w0
    return perm


def sell_layout(lens, C: int, sigma: int, exclude=None, group: int = 1) -> dict:
    """SELL-C-sigma layout sizes.

    ``exclude``: rows that are stored elsewhere (long rows); they count as empty here.
    ``group``: slice widths are rounded up to a multiple of it (the column-grouped
    layout for ``group`` threads per row stores whole groups).
    Returned keys:
      perm            sorted position -> original row (length n)
      sorted_lens     lengths in sorted order (excluded rows are 0)
      widths          per-slice width = longest row in the slice, rounded up to whole groups (n_slices)
      slice_ptr       int64 exclusive scan of C * width (n_slices + 1)
      padded_entries  sum over real rows of their slice's width
      allocated_slots sum over slices of C * width (includes the rows that pad n to a multiple of C)
    """
    lens = np.asarray(lens, dtype=np.int64).copy()
    if exclude is not None and len(exclude):
        lens[np.asarray(exclude, dtype=np.int64)] = 0
    n = lens.size
    perm = sell_order(lens, sigma)
    sorted_lens = lens[perm]
    n_slices = -(-n // C)
    padded = np.zeros(n_slices * C, dtype=np.int64)
    padded[:n] = sorted_lens
    widths = padded.reshape(n_slices, C).max(axis=1) if n_slices else np.zeros(0, np.int64)
    widths = -(-widths // group) * group
    slice_ptr = np.zeros(n_slices + 1, dtype=np.int64)
    np.cumsum(widths * C, out=slice_ptr[1:])
    rows_in_slice = np.minimum(C, n - np.arange(n_slices) * C)
    return {
        "perm": perm,
        "sorted_lens": sorted_lens,
        "widths": widths,
        "slice_ptr": slice_ptr,
        "padded_entries": int((widths * rows_in_slice).sum()),
        "allocated_slots": int(slice_ptr[-1]),
    }


def slot_offset(q, j, stride: int, group: int = 1, interleaved: bool = False):
    """Offset, inside its slice, of entry j of the row at in-slice position q.

    Column-major (the ELLPACK / SELL layout of the spMVM paper, Fig. 1): entry j of all
    rows of the slice is contiguous, offset j * stride + q.  Column-grouped (the AMD
    rearrangement the load-balancing SpMV paper describes, for ``group`` threads per
    row): the slice is walked group of columns by group of columns, then row by row,
    then column by column inside the group, i.e. entries j of row q with the same
    j // group sit side by side: offset ((j // group) * stride + q) * group + j % group.
    """
    q = np.asarray(q, dtype=np.int64)
    j = np.asarray(j, dtype=np.int64)
    if not interleaved:
        return j * stride + q
    return ((j // group) * stride + q) * group + j % group


def sell_slots(csr, C: int, sigma: int, exclude=None, group: int = 1, interleaved: bool = False,
               ell_ld: int | None = None, group_val: int | None = None, round_to: int | None = None) -> tuple:
    """The slot arrays (column, value) of a sliced layout built from ``csr``.

    SELL (``ell_ld`` None): slices of C sorted positions with ``sell_layout`` widths.
    ELLPACK (``ell_ld`` given): one slice, rows in natural order, leading dimension
    ``ell_ld``, width = the longest stored row.  Widths are rounded up to whole groups
    in the column-grouped (interleaved) layout only (to ``round_to`` when given).
    ``group_val``: the value array grouped differently from the index array (the
    16-byte vector layout: indices in groups of 4, values in groups of 16 bytes).
    Excluded rows and padding slots hold column 0 and value 0.
    """
    lens = row_lengths(csr.row_ptr)
    if round_to is None:
        round_to = group if interleaved else 1  # only the column-grouped layout stores whole groups
    gv = group if group_val is None else group_val
    if ell_ld is None:
        lay = sell_layout(lens, C, sigma, exclude=exclude, group=round_to)
        perm, stored, starts, stride = lay["perm"], lay["sorted_lens"], lay["slice_ptr"], C
        total = int(starts[-1])
        pos = np.arange(perm.size, dtype=np.int64)
        base = starts[pos // C]
        q = pos % C
    else:
        stored = lens.astype(np.int64).copy()
        if exclude is not None and len(exclude):
            stored[np.asarray(exclude, dtype=np.int64)] = 0
        perm = np.arange(csr.n, dtype=np.int64)
        width = int(stored.max()) if stored.size else 0
        width = -(-width // round_to) * round_to
        stride, total = ell_ld, ell_ld * width
        base = np.zeros(csr.n, dtype=np.int64)
        q = np.arange(csr.n, dtype=np.int64)
    col = np.zeros(total, dtype=np.int32)
    val = np.zeros(total, dtype=csr.vals.dtype)
    reps = stored.astype(np.int64)
    P = np.repeat(np.arange(perm.size), reps)
    J = np.arange(P.size) - np.repeat(np.cumsum(reps) - reps, reps)
    src = csr.row_ptr[perm[P]].astype(np.int64) + J
    col[base[P] + slot_offset(q[P], J, stride, group, interleaved)] = csr.col_idx[src]
    val[base[P] + slot_offset(q[P], J, stride, gv, interleaved)] = csr.vals[src]
    return col, val


def ellpack_entries(lens) -> int:
    """ELLPACK / ELLPACK-R storage: N x max row length."""
    lens = np.asarray(lens, dtype=np.int64)
    return int(lens.size * (lens.max() if lens.size else 0))


def pjds_entries(lens, b_r: int) -> int:
    """pJDS storage: rows sorted longest first, blocks of b_r rows padded to their longest row."""
    lens = np.asarray(lens, dtype=np.int64)
    return sell_layout(lens, b_r, max(lens.size, 1))["padded_entries"]


def ell_leading_dim(n: int, multiple: int = 256) -> int:
    """Leading dimension of the HYB/HEC ELL part: n rounded up to a multiple of 32 (256 here)."""
    return -(-n // multiple) * multiple if n else 0


def hyb_modeled_bytes(lens, K: int, value_bytes: int, ld: int, c: float = 1.0) -> float:
    """Bytes to stream the HYB parts: ELL slots (value + int32 column) for every row slot up
    to width K, plus c * (value + int32 row + int32 column) per spilled entry."""
    lens = np.asarray(lens, dtype=np.int64)
    spill = np.maximum(lens - K, 0).sum()
    return ld * K * (value_bytes + 4) + c * (value_bytes + 8) * float(spill)


def hyb_width(lens, value_bytes: int, ld: int | None = None, c: float = 1.0, k_cap: int | None = None) -> int:
    """ELL width K of the HYB split chosen from the row-length histogram.

    Widening the ELL part by one column costs ld * (value_bytes + 4) bytes and removes
    c * (value_bytes + 8) bytes for every row still longer than K, so the byte model is
    convex in K and its smallest minimiser is the smallest K with
        c * (value_bytes + 8) * #{i : len_i > K} <= ld * (value_bytes + 4).
    The result is capped at ``k_cap``.
    """
    lens = np.asarray(lens, dtype=np.int64)
    n = lens.size
    if ld is None:
        ld = ell_leading_dim(n)
    maxlen = int(lens.max()) if n else 0
    hist = np.bincount(lens, minlength=maxlen + 1)
    longer = n - np.cumsum(hist)  # longer[K] = #{len > K}
    K = 0
    while K < maxlen and c * (value_bytes + 8) * longer[K] > ld * (value_bytes + 4):
        K += 1
    if k_cap is not None:
        K = min(K, int(k_cap))
    return K


def hyb_split(lens, K: int) -> dict:
    """ELL part widths (min(len, K)) and the spill size of the HYB split."""
    lens = np.asarray(lens, dtype=np.int64)
    ell = np.minimum(lens, K)
    spill = lens - ell
    return {"ell_lens": ell, "spill_lens": spill, "spill_nnz": int(spill.sum()),
            "spill_rows": np.nonzero(spill > 0)[0]}
