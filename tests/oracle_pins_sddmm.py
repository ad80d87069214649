"""Pins of the SDDMM and FusedMM oracles to facts independent of them.

SDDMM (page "Performance Optimization of Deep Learning Sparse Matrix Kernels
on Intel Max Series GPU", SDDMM section, Algorithm 1): out[p] = C_i . B_j for
every stored (i, j) of A.  FusedMM (same page, Fig. 6, Algorithm 3):
E_i = sum_j (C_i . B_j) D_j over the stored j of row i.

Each pin takes callables ``sddmm(rowptr, colind, C, B) -> (out, S)`` and
``fusedmm(rowptr, colind, C, B, D) -> (E, S)`` and raises AssertionError on a
disagreement with: numpy's dense float64 matmul masked by the pattern, closed
forms (dense pattern, identity pattern, zero B), int64 matmuls on integer
data, a hand-worked 2x2 example, and (FusedMM) the composition of the SDDMM
oracle with the independently pinned SpMM oracle on integer data.
"""
from __future__ import annotations

import numpy as np

import oracle
from csr_spmm_02_gb300 import gen


def _pattern(rng, M, K, mean_row=4, empty_frac=0.25, duplicates=False):
    p = gen.random_csr(rng, M, K, 1, mean_row=mean_row, empty_frac=empty_frac, long_rows=[(0, K)],
                       duplicates=duplicates)
    return p.rowptr, p.colind


def _rows(rowptr):
    return np.repeat(np.arange(len(rowptr) - 1), np.diff(rowptr))


def pin_sddmm_dense_masked(sddmm, fusedmm):
    rng = np.random.default_rng(21)
    for N in (1, 4, 17, 64):
        M, K = int(rng.integers(1, 50)), int(rng.integers(1, 50))
        rowptr, colind = _pattern(rng, M, K, duplicates=True)
        C = rng.standard_normal((M, N)).astype(np.float32)
        B = rng.standard_normal((K, N)).astype(np.float32)
        out, S = sddmm(rowptr, colind, C, B)
        full = C.astype(np.float64) @ B.astype(np.float64).T
        mag = np.abs(C.astype(np.float64)) @ np.abs(B.astype(np.float64)).T
        r = _rows(rowptr)
        ref, refS = full[r, colind], mag[r, colind]
        assert np.all(np.abs(out - ref) <= 1e-12 * refS + 1e-300), f"SDDMM vs masked dense product (N={N})"
        assert np.all(np.abs(S - refS) <= 1e-12 * refS + 1e-300)


def pin_sddmm_closed_forms(sddmm, fusedmm):
    rng = np.random.default_rng(22)
    M, K, N = 7, 5, 9
    C = rng.integers(-3, 4, (M, N)).astype(np.float32)
    B = rng.integers(-3, 4, (K, N)).astype(np.float32)
    # dense pattern: every entry of C . B^T, exactly (small integers)
    rowptr = (np.arange(M + 1) * K).astype(np.int32)
    colind = np.tile(np.arange(K), M).astype(np.int32)
    out, _ = sddmm(rowptr, colind, C, B)
    assert np.array_equal(out.reshape(M, K), C.astype(np.int64) @ B.astype(np.int64).T), "dense pattern"
    # identity pattern with B = C: squared row norms
    rp, ci, _ = gen.identity_csr(M)
    out, _ = sddmm(rp, ci, C, C)
    assert np.array_equal(out, (C.astype(np.int64) ** 2).sum(axis=1)), "identity pattern: squared norms"


def pin_sddmm_hand_2x2(sddmm, fusedmm):
    # A's pattern: (0,1), (1,0), (1,1).  C = [[1,2],[3,4]], B = [[5,6],[7,8]].
    # out(0,1) = 1*7 + 2*8 = 23; out(1,0) = 3*5 + 4*6 = 39; out(1,1) = 3*7 + 4*8 = 53.
    rowptr = np.array([0, 1, 3], np.int32)
    colind = np.array([1, 0, 1], np.int32)
    C = np.array([[1, 2], [3, 4]], np.float32)
    B = np.array([[5, 6], [7, 8]], np.float32)
    out, _ = sddmm(rowptr, colind, C, B)
    assert list(out) == [23.0, 39.0, 53.0]
    # FusedMM with D = [[1,0],[0,1]] (identity): E_0 = 23*[0,1]; E_1 = 39*[1,0] + 53*[0,1].
    E, _ = fusedmm(rowptr, colind, C, B, np.eye(2, dtype=np.float32))
    assert E.tolist() == [[0.0, 23.0], [39.0, 53.0]]


def pin_fusedmm_dense(sddmm, fusedmm):
    rng = np.random.default_rng(23)
    for N in (1, 5, 32):
        M, K = int(rng.integers(1, 40)), int(rng.integers(1, 40))
        rowptr, colind = _pattern(rng, M, K, duplicates=True)
        C = rng.standard_normal((M, N)).astype(np.float32)
        B = rng.standard_normal((K, N)).astype(np.float32)
        D = rng.standard_normal((K, N)).astype(np.float32)
        E, S = fusedmm(rowptr, colind, C, B, D)
        r = _rows(rowptr)
        full = C.astype(np.float64) @ B.astype(np.float64).T
        Amask = np.zeros((M, K))
        np.add.at(Amask, (r, colind), full[r, colind])  # duplicates add their sampled value twice
        ref = Amask @ D.astype(np.float64)
        Aabs = np.zeros((M, K))
        np.add.at(Aabs, (r, colind), np.abs(full[r, colind]))
        refS = Aabs @ np.abs(D.astype(np.float64))
        assert np.all(np.abs(E - ref) <= 1e-11 * refS + 1e-300), f"FusedMM vs dense (N={N})"
        assert np.all(np.abs(S - refS) <= 1e-11 * refS + 1e-300)


def pin_fusedmm_special(sddmm, fusedmm):
    rng = np.random.default_rng(24)
    M, K, N = 12, 9, 6
    rowptr, colind = _pattern(rng, M, K)
    C = rng.standard_normal((M, N)).astype(np.float32)
    D = rng.standard_normal((K, N)).astype(np.float32)
    E, _ = fusedmm(rowptr, colind, C, np.zeros((K, N), np.float32), D)
    assert not E.any(), "B = 0 gives E = 0"
    # identity pattern: E_i = (C_i . B_i) D_i
    C = rng.integers(-3, 4, (M, N)).astype(np.float32)
    B = rng.integers(-3, 4, (M, N)).astype(np.float32)
    D = rng.integers(-3, 4, (M, N)).astype(np.float32)
    rp, ci, _ = gen.identity_csr(M)
    E, _ = fusedmm(rp, ci, C, B, D)
    dots = (C.astype(np.int64) * B.astype(np.int64)).sum(axis=1)
    assert np.array_equal(E, dots[:, None] * D.astype(np.int64)), "identity pattern"


def pin_fusedmm_is_sddmm_then_spmm(sddmm, fusedmm):
    """Integer data: E equals the SpMM oracle applied to the SDDMM oracle's values (all exact)."""
    rng = np.random.default_rng(25)
    M, K, N = 30, 25, 7
    rowptr, colind = _pattern(rng, M, K, mean_row=5, duplicates=True)
    C = rng.integers(-2, 3, (M, N)).astype(np.float32)
    B = rng.integers(-2, 3, (K, N)).astype(np.float32)
    D = rng.integers(-3, 4, (K, N)).astype(np.float32)
    a, _ = sddmm(rowptr, colind, C, B)
    E_ref, _ = oracle.spmm_reference(rowptr, colind, a.astype(np.float32), D)
    E, _ = fusedmm(rowptr, colind, C, B, D)
    assert np.array_equal(E, E_ref), "FusedMM = SpMM(SDDMM values)"
    r = _rows(rowptr)
    Ai = np.zeros((M, K), np.int64)
    np.add.at(Ai, (r, colind), (C.astype(np.int64) @ B.astype(np.int64).T)[r, colind])
    assert np.array_equal(E, (Ai @ D.astype(np.int64)).astype(np.float64)), "FusedMM vs int64"


ALL_PINS = [pin_sddmm_dense_masked, pin_sddmm_closed_forms, pin_sddmm_hand_2x2, pin_fusedmm_dense,
            pin_fusedmm_special, pin_fusedmm_is_sddmm_then_spmm]


def callables(library=None):
    def sddmm(rowptr, colind, C, B):
        return oracle.sddmm_reference(rowptr, colind, C, B, library=library)

    def fusedmm(rowptr, colind, C, B, D):
        return oracle.fusedmm_reference(rowptr, colind, C, B, D, library=library)
    return sddmm, fusedmm


def failing_pins(library=None):
    sddmm, fusedmm = callables(library)
    bad = []
    for pin in ALL_PINS:
        try:
            pin(sddmm, fusedmm)
        except (AssertionError, ValueError):
            bad.append(pin.__name__)
    return bad
