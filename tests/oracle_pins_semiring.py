"""Pins of the semiring SpMM oracle to facts independent of it.

Definition (page "Sgap: Towards Efficient Sparse Tensor Algebra Compilation
for GPU", sparse-dense hybrid algebra, Eq. 3): C[i, n] is the (+)-reduction,
over row i's stored entries, of vals[p] (x) B[colind[p], n]; (+) in
{sum, min, max}, (x) in {multiply, add}; an empty row gives (+)'s identity.

Each pin takes ``semiring(rowptr, colind, vals, B, add, mul) -> (C, S)`` and
raises AssertionError on a disagreement with: a hand-worked 3x2 example;
numpy ufunc reductions over each row's entry products (``np.minimum.reduceat``
and friends, duplicates and empty rows included); a densified float64 matmul
for sum/multiply; closed forms (B = 1 under max/multiply gives each row's
largest value, B = 0 under min/add its smallest); and single-source shortest
paths: iterating x <- min(x, A (min,+) x) from a source reaches the distances
that scipy's Dijkstra computes (integer weights, so both are exact).
"""
from __future__ import annotations

import numpy as np

import oracle
from csr_spmm_02_gb300 import gen

IDENTITY = {"sum": 0.0, "min": np.inf, "max": -np.inf}
OPS = [(a, m) for a in ("sum", "min", "max") for m in ("mul", "add")]


def _pattern(rng, M, K, mean_row=4, empty_frac=0.3, duplicates=True):
    p = gen.random_csr(rng, M, K, 1, mean_row=mean_row, max_row=K, empty_frac=empty_frac,
                       duplicates=duplicates, sort_cols=False)
    return p.rowptr, p.colind


def _rowwise(rowptr, colind, vals, B, add, mul):
    """Per-entry values reduced per row with numpy ufuncs (empty rows: identity)."""
    B64 = B.astype(np.float64)
    a = vals.astype(np.float64)[:, None]
    T = a * B64[colind] if mul == "mul" else a + B64[colind]
    M, N = len(rowptr) - 1, B.shape[1]
    out = np.full((M, N), IDENTITY[add])
    lens = np.diff(rowptr)
    nz = np.flatnonzero(lens > 0)
    if len(nz):
        ufunc = {"sum": np.add, "min": np.minimum, "max": np.maximum}[add]
        out[nz] = ufunc.reduceat(T, rowptr[nz], axis=0)
    return out


def pin_hand_3x2(semiring):
    # Rows: 0 -> (col 0, 1), (col 1, 2); 1 -> empty; 2 -> (col 1, 3).  B = [[1, 5], [2, -1]].
    rowptr = np.array([0, 2, 2, 3], np.int32)
    colind = np.array([0, 1, 1], np.int32)
    vals = np.array([1, 2, 3], np.float32)
    B = np.array([[1, 5], [2, -1]], np.float32)
    inf = np.inf
    expect = {
        ("sum", "mul"): [[5, 3], [0, 0], [6, -3]],     # 1*1+2*2, 1*5+2*(-1)
        ("sum", "add"): [[6, 7], [0, 0], [5, 2]],      # (1+1)+(2+2), (1+5)+(2-1)
        ("min", "mul"): [[1, -2], [inf, inf], [6, -3]],
        ("min", "add"): [[2, 1], [inf, inf], [5, 2]],
        ("max", "mul"): [[4, 5], [-inf, -inf], [6, -3]],
        ("max", "add"): [[4, 6], [-inf, -inf], [5, 2]],
    }
    for (add, mul), e in expect.items():
        C, _ = semiring(rowptr, colind, vals, B, add, mul)
        assert np.array_equal(C, np.array(e, np.float64)), (add, mul, C)


def pin_rowwise_ufuncs(semiring):
    rng = np.random.default_rng(31)
    for add, mul in OPS:
        for N in (1, 3, 8):
            M, K = int(rng.integers(1, 60)), int(rng.integers(1, 60))
            rowptr, colind = _pattern(rng, M, K)
            vals = rng.standard_normal(len(colind)).astype(np.float32)
            B = rng.standard_normal((K, N)).astype(np.float32)
            C, S = semiring(rowptr, colind, vals, B, add, mul)
            ref = _rowwise(rowptr, colind, vals, B, add, mul)
            if add == "sum":
                assert np.allclose(C, ref, rtol=1e-12, atol=1e-12), (add, mul, N)
                mag = np.zeros_like(C)
                for i in range(M):
                    for p in range(rowptr[i], rowptr[i + 1]):
                        t = vals[p] * B[colind[p]].astype(np.float64) if mul == "mul" else \
                            vals[p] + B[colind[p]].astype(np.float64)
                        mag[i] += np.abs(t)
                assert np.allclose(S, mag, rtol=1e-12, atol=1e-12)
            else:
                assert np.array_equal(C, ref), (add, mul, N)


def pin_sum_mul_is_matmul(semiring):
    rng = np.random.default_rng(32)
    M, K, N = 37, 23, 5
    rowptr, colind = _pattern(rng, M, K)
    vals = rng.standard_normal(len(colind)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    A = np.zeros((M, K))
    rows = np.repeat(np.arange(M), np.diff(rowptr))
    np.add.at(A, (rows, colind), vals.astype(np.float64))
    C, _ = semiring(rowptr, colind, vals, B, "sum", "mul")
    assert np.allclose(C, A @ B.astype(np.float64), rtol=1e-12, atol=1e-12)


def pin_closed_forms(semiring):
    rng = np.random.default_rng(33)
    M, K, N = 40, 30, 3
    rowptr, colind = _pattern(rng, M, K)
    vals = rng.standard_normal(len(colind)).astype(np.float32)
    lens = np.diff(rowptr)
    C, _ = semiring(rowptr, colind, vals, np.ones((K, N), np.float32), "max", "mul")
    C2, _ = semiring(rowptr, colind, vals, np.zeros((K, N), np.float32), "min", "add")
    for i in range(M):
        seg = vals[rowptr[i]:rowptr[i + 1]].astype(np.float64)
        assert np.all(C[i] == (seg.max() if lens[i] else -np.inf))
        assert np.all(C2[i] == (seg.min() if lens[i] else np.inf))


def pin_shortest_paths(semiring):
    import scipy.sparse as sp
    from scipy.sparse.csgraph import dijkstra
    rng = np.random.default_rng(34)
    n = 60
    src, dst = rng.integers(0, n, 300), rng.integers(0, n, 300)
    keep = src != dst
    src, dst = src[keep], dst[keep]
    _, first = np.unique(src * n + dst, return_index=True)  # distinct edges (scipy sums repeats)
    src, dst = src[first], dst[first]
    w = rng.integers(1, 20, len(src)).astype(np.float32)
    # row i of A lists the edges j -> i with their weights: (A (min,+) x)[i] = min_j w_ji + x[j]
    order = np.lexsort((src, dst))
    rowptr = np.zeros(n + 1, np.int32)
    np.add.at(rowptr, dst[order] + 1, 1)
    rowptr = np.cumsum(rowptr).astype(np.int32)
    colind = src[order].astype(np.int32)
    vals = w[order]
    x = np.full((n, 1), np.inf, np.float32)
    x[0, 0] = 0.0
    for _ in range(n):
        y, _ = semiring(rowptr, colind, vals, x, "min", "add")
        x = np.minimum(x, y).astype(np.float32)
    G = sp.coo_matrix((w.astype(np.float64), (src, dst)), shape=(n, n)).tocsr()
    ref = dijkstra(G, directed=True, indices=0)
    assert np.array_equal(x[:, 0].astype(np.float64), ref), "Bellman-Ford by (min,+) SpMM != Dijkstra"


ALL_PINS = [pin_hand_3x2, pin_rowwise_ufuncs, pin_sum_mul_is_matmul, pin_closed_forms, pin_shortest_paths]


def callables(library=None):
    def semiring(rowptr, colind, vals, B, add, mul):
        return oracle.semiring_reference(rowptr, colind, vals, B, add, mul, library=library)
    return semiring


def failing_pins(library=None):
    semiring = callables(library)
    bad = []
    for pin in ALL_PINS:
        try:
            pin(semiring)
        except (AssertionError, ValueError):
            bad.append(pin.__name__)
    return bad
