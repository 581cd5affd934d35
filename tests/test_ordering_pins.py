"""Pins for the symmetric orderings and the permuted basis (oracle/ordering.py):
dense P A P^T, the stable row-length sort, Cuthill-McKee orders derived by hand from
its definition, closed forms on paths, stars and grids, a second formulation of the
same ordering (breadth-first levels, each ordered by earliest parent then degree and
index), and bandwidth against scipy's reverse Cuthill-McKee."""
import numpy as np
import pytest

from oracle import ordering
from workloads import CSR, laplacian_1d, laplacian_2d, laplacian_3d, random_csr


def dense(csr):
    D = np.zeros((csr.n, csr.n))
    for i in range(csr.n):
        for k in range(csr.row_ptr[i], csr.row_ptr[i + 1]):
            D[i, csr.col_idx[k]] += csr.vals[k]
    return D


def from_edges(n, edges, diag=True):
    rows = [[i] if diag else [] for i in range(n)]
    for u, v in edges:
        rows[u].append(v)
        rows[v].append(u)
    row_ptr = np.zeros(n + 1, np.int32)
    row_ptr[1:] = np.cumsum([len(r) for r in rows])
    cols = np.array([c for r in rows for c in sorted(r)], np.int32)
    return CSR(n, row_ptr, cols, np.ones(cols.size))


def relabel(csr, seed):
    perm = np.random.default_rng(seed).permutation(csr.n)
    return ordering.symmetric_permute(csr, perm)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_symmetric_permute_is_dense_pap(seed):
    csr = random_csr(40, density=0.15, seed=seed, duplicates=True, unsorted=True, empty_row_fraction=0.1)
    perm = np.random.default_rng(seed + 10).permutation(csr.n)
    B = ordering.symmetric_permute(csr, perm)
    P = np.eye(csr.n)[perm]
    assert np.array_equal(dense(B), P @ dense(csr) @ P.T)
    # in-row order of A is kept
    for i in range(csr.n):
        a = csr.vals[csr.row_ptr[perm[i]]:csr.row_ptr[perm[i] + 1]]
        assert np.array_equal(B.vals[B.row_ptr[i]:B.row_ptr[i + 1]], a)


def test_row_length_order_stable_descending():
    csr = random_csr(300, density=0.03, seed=4, empty_row_fraction=0.2, full_rows=2)
    lens = np.diff(csr.row_ptr)
    perm = ordering.row_length_order(csr)
    assert sorted(perm.tolist()) == list(range(csr.n))
    expect = sorted(range(csr.n), key=lambda i: (-lens[i], i))
    assert perm.tolist() == expect


def test_cuthill_mckee_by_hand():
    """0-{1,2,3}, 1-{4,5}, 2-6, plus vertex 7 alone.  Degrees 3,3,2,1,1,1,1,0.  Vertex 7
    (degree 0) first; start at the least (degree, index) vertex, 3; 3 -> 0; 0's
    neighbours by degree: 2 (2), 1 (3); then 2 -> 6; 1 -> 4, 5."""
    csr = from_edges(8, [(0, 1), (0, 2), (0, 3), (1, 4), (1, 5), (2, 6)])
    assert ordering.cuthill_mckee(csr).tolist() == [7, 3, 0, 2, 1, 6, 4, 5]
    assert ordering.reverse_cuthill_mckee(csr).tolist() == [5, 4, 6, 1, 2, 0, 3, 7]


def test_star_graph():
    """Centre 5 with leaves 0..4, 6..9: start at leaf 0, then the centre, then the other
    leaves in index order (all of degree 1)."""
    csr = from_edges(10, [(5, v) for v in range(10) if v != 5])
    assert ordering.cuthill_mckee(csr).tolist() == [0, 5, 1, 2, 3, 4, 6, 7, 8, 9]


@pytest.mark.parametrize("seed", [3, 4])
def test_shuffled_path_becomes_tridiagonal(seed):
    B = relabel(laplacian_1d(200), seed)
    R = ordering.symmetric_permute(B, ordering.reverse_cuthill_mckee(B))
    assert ordering.bandwidth(R) == 1


def test_components_in_order():
    """Two paths 0-2-4 and 1-3 and isolated 5: isolated first, then each component from its
    least (degree, index) vertex: 0 (deg 1) runs 0, 2, 4; then 1 runs 1, 3."""
    csr = from_edges(6, [(0, 2), (2, 4), (1, 3)])
    assert ordering.cuthill_mckee(csr).tolist() == [5, 0, 2, 4, 1, 3]


def test_nonsymmetric_pattern_uses_a_plus_at():
    # entries only above the diagonal: 0->1, 1->2 ; the graph is still the path 0-1-2
    csr = CSR(3, np.array([0, 1, 2, 2], np.int32), np.array([1, 2], np.int32), np.ones(2))
    ptr, adj = ordering.symmetric_graph(csr)
    assert ptr.tolist() == [0, 1, 3, 4] and adj.tolist() == [1, 0, 2, 1]
    assert ordering.cuthill_mckee(csr).tolist() == [0, 1, 2]


def levels_formulation(csr):
    """The same ordering built level by level: every unvisited neighbour of the current
    level is claimed by its earliest-ordered neighbour there, and the next level is
    sorted by (claiming position, degree, index)."""
    ptr, adj = ordering.symmetric_graph(csr)
    n = csr.n
    deg = np.diff(ptr)
    pos = -np.ones(n, np.int64)
    order = list(np.nonzero(deg == 0)[0])
    for i, v in enumerate(order):
        pos[v] = i
    for start in sorted(range(n), key=lambda v: (deg[v], v)):
        if pos[start] >= 0:
            continue
        pos[start] = len(order)
        order.append(start)
        lo, hi = len(order) - 1, len(order)
        while lo < hi:
            claim = {}
            for i in range(lo, hi):
                u = order[i]
                for v in adj[ptr[u]:ptr[u + 1]]:
                    if pos[v] < 0:
                        claim[int(v)] = min(claim.get(int(v), i), i)
            nxt = sorted(claim, key=lambda v: (claim[v], deg[v], v))
            for v in nxt:
                pos[v] = len(order)
                order.append(v)
            lo, hi = hi, len(order)
    return np.array(order)


@pytest.mark.parametrize("seed", range(6))
def test_level_formulation_agrees(seed):
    csr = random_csr(120, density=0.02 + 0.01 * seed, seed=seed, empty_row_fraction=0.05)
    assert np.array_equal(levels_formulation(csr), ordering.cuthill_mckee(csr))


@pytest.mark.parametrize("make", [lambda: laplacian_2d(30, 20), lambda: laplacian_3d(9, 8, 7)])
def test_grid_bandwidth_against_scipy(make):
    from scipy.sparse import csr_matrix
    from scipy.sparse.csgraph import reverse_cuthill_mckee as scipy_rcm

    B = relabel(make(), 5)
    ours = ordering.bandwidth(ordering.symmetric_permute(B, ordering.reverse_cuthill_mckee(B)))
    m = csr_matrix((B.vals, B.col_idx, B.row_ptr), shape=(B.n, B.n))
    theirs = ordering.bandwidth(ordering.symmetric_permute(B, np.asarray(scipy_rcm(m, symmetric_mode=True))))
    assert ours <= max(theirs * 5 // 4, theirs + 2)
    assert ours < ordering.bandwidth(B) // 4
