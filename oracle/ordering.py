"""Symmetric orderings and the permuted basis -- oracle, TEST INFRASTRUCTURE ONLY.

The GPGPU spMVM paper (arXiv 1112.5588, pJDS section) notes that its sorted format
works in a permuted basis, and that for Krylov solvers the permutation is applied once
before and once after the iteration, while the iteration itself runs on permuted
vectors; it also notes that sorting rows can destroy structure and with it the cache
reuse of the right-hand side.  The permuted basis here is B = P A P^T: row and column i
of B are row and column perm[i] of A (perm maps new index -> original index).

Orderings (perm, new -> old):
* ``row_length_order``: rows by length, longest first, ties in index order (the pJDS
  sort over the whole matrix).
* ``cuthill_mckee`` / ``reverse_cuthill_mckee``: the Cuthill-McKee (1969) breadth-first
  ordering of the graph of A + A^T (an edge u-v for every stored entry off the
  diagonal, either way round; degrees count distinct neighbours).  The pages give no
  ordering of this kind; the definition followed, written as the textbook queue
  algorithm:
    - vertices of degree 0 first, in index order;
    - then, while vertices remain, start a component at the unvisited vertex of least
      (degree, index) and run the queue: take the next vertex of the ordering, append
      its unvisited neighbours sorted by (degree, index);
    - reverse Cuthill-McKee is that ordering reversed.

Pinned by ``tests/test_ordering_pins.py``.
"""
from __future__ import annotations

from collections import deque

import numpy as np


def symmetric_graph(csr):
    """Adjacency lists (sorted, distinct, no self loops) of the graph of A + A^T."""
    n = csr.n
    rows = np.repeat(np.arange(n, dtype=np.int64), np.diff(csr.row_ptr.astype(np.int64)))
    cols = csr.col_idx.astype(np.int64)
    off = rows != cols
    u = np.concatenate([rows[off], cols[off]])
    v = np.concatenate([cols[off], rows[off]])
    key = np.unique(u * n + v)
    u, v = key // n, key % n
    ptr = np.zeros(n + 1, dtype=np.int64)
    np.add.at(ptr, u + 1, 1)
    ptr = np.cumsum(ptr)
    return ptr, v


def row_length_order(csr) -> np.ndarray:
    lens = np.diff(csr.row_ptr.astype(np.int64))
    return np.argsort(-lens, kind="stable").astype(np.int64)


def cuthill_mckee(csr) -> np.ndarray:
    ptr, adj = symmetric_graph(csr)
    n = csr.n
    deg = np.diff(ptr)
    visited = np.zeros(n, dtype=bool)
    order = [int(v) for v in np.nonzero(deg == 0)[0]]
    visited[order] = True
    by_deg_index = np.lexsort((np.arange(n), deg))  # least (degree, index) first
    k = 0
    while len(order) < n:
        while visited[by_deg_index[k]]:
            k += 1
        start = int(by_deg_index[k])
        visited[start] = True
        order.append(start)
        queue = deque([start])
        while queue:
            u = queue.popleft()
            nb = [int(v) for v in adj[ptr[u]:ptr[u + 1]] if not visited[v]]
            nb.sort(key=lambda v: (deg[v], v))
            for v in nb:
                visited[v] = True
                order.append(v)
                queue.append(v)
    return np.array(order, dtype=np.int64)


def reverse_cuthill_mckee(csr) -> np.ndarray:
    return cuthill_mckee(csr)[::-1].copy()


def symmetric_permute(csr, perm):
    """B = P A P^T as a CSR of the same class: row i of B is row perm[i] of A, with every
    column c renamed to inv[c] (inv = inverse of perm), entries in A's in-row order."""
    perm = np.asarray(perm, dtype=np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    lens = np.diff(csr.row_ptr.astype(np.int64))[perm]
    row_ptr = np.zeros(csr.n + 1, dtype=np.int64)
    np.cumsum(lens, out=row_ptr[1:])
    starts = csr.row_ptr.astype(np.int64)[perm]
    idx = np.repeat(starts - row_ptr[:-1], lens) + np.arange(int(row_ptr[-1]))
    return type(csr)(csr.n, row_ptr.astype(np.int32), inv[csr.col_idx[idx]].astype(np.int32), csr.vals[idx].copy())


def bandwidth(csr) -> int:
    """max |i - j| over stored entries."""
    rows = np.repeat(np.arange(csr.n, dtype=np.int64), np.diff(csr.row_ptr.astype(np.int64)))
    return int(np.abs(rows - csr.col_idx.astype(np.int64)).max()) if rows.size else 0
