"""Checks that pin the CPU oracle to facts independent of the oracle itself.

Each ``pin_*`` function takes an oracle callable
``fn(rowptr, colind, vals, B, b_dtype="f32", rows=None) -> (C, S)`` and raises
AssertionError when the oracle disagrees with:

* a textbook routine -- the sparse matrix densified by scatter-add and
  multiplied with numpy's dense float64 matmul, or an int64 matmul for
  integer data;
* brute force over every 0/1 sparsity pattern of a 3x3 matrix;
* closed forms -- identity, permutation and power-of-two scaled identity
  (exact), a column of ones (row sums), an indicator column (a column of A),
  the 2^24 + 1 sum that only a double accumulator keeps;
* the hand-worked 4x4 example in ``tests/golden/hand_4x4.txt``;
* invariants -- linearity in the values, row-subset consistency;
* a library routine for bf16 decoding (torch's bfloat16 -> float32).

The SpMM definition being pinned: C[i, n] = sum over the nonzeros p of row i
of vals[p] * B[colind[p], n] (page "Performance Optimization of Deep Learning
Sparse Matrix Kernels on Intel Max Series GPU", SPMM section, Algorithm 2);
S is the same sum of absolute products.
"""
from __future__ import annotations

import itertools
import os

import numpy as np

from csr_spmm_02_gb300 import gen

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def densify(rowptr, colind, vals, K, absolute=False):
    """Dense float64 A from CSR by scatter-add (duplicates summed)."""
    M = len(rowptr) - 1
    A = np.zeros((M, K), dtype=np.float64)
    rows = np.repeat(np.arange(M), np.diff(rowptr))
    v = np.abs(vals.astype(np.float64)) if absolute else vals.astype(np.float64)
    np.add.at(A, (rows, colind.astype(np.int64)), v)
    return A


def load_golden_hand_4x4():
    lines = [ln.strip() for ln in open(os.path.join(GOLDEN, "hand_4x4.txt")) if ln.strip() and not ln.startswith("#")]
    out, it = {}, iter(lines)
    for ln in it:
        key, rest = ln.split(":", 1)
        nums = rest.split()
        if key in ("rowptr", "colind", "vals"):
            out[key] = np.array([float(x) for x in nums])
        else:
            r, c = int(nums[0]), int(nums[1])
            out[key] = np.array([[float(x) for x in next(it).split()] for _ in range(r)]).reshape(r, c)
    return out


def _as_f64(B, b_dtype):
    if b_dtype == "f32":
        return B.astype(np.float64)
    import torch
    return torch.from_numpy(B.view(np.int16).copy()).view(torch.bfloat16).float().numpy().astype(np.float64)


# ----------------------------------------------------------------------------
def pin_dense_matmul(fn):
    """Random tiny matrices (empty rows, a full row, duplicates, unsorted) vs numpy matmul."""
    rng = np.random.default_rng(123)
    for trial, N in enumerate((1, 3, 4, 8, 33)):
        M, K = int(rng.integers(1, 65)), int(rng.integers(1, 65))
        p = gen.random_csr(rng, M, K, N, mean_row=5, empty_frac=0.25,
                           long_rows=[(0, K)], duplicates=(trial % 2 == 1), sort_cols=(trial % 3 != 0))
        C, S = fn(p.rowptr, p.colind, p.vals, p.B)
        B64 = p.B.astype(np.float64)
        Cd = densify(p.rowptr, p.colind, p.vals, K) @ B64
        Sd = densify(p.rowptr, p.colind, p.vals, K, absolute=True) @ np.abs(B64)
        tol = 1e-12 * Sd + 1e-300
        assert C.shape == (M, N) and S.shape == (M, N)
        assert np.all(np.abs(C - Cd) <= tol), f"C differs from dense matmul (trial {trial})"
        assert np.all(np.abs(S - Sd) <= tol), f"S differs from |A| @ |B| (trial {trial})"


def pin_bruteforce_3x3(fn):
    """Every 0/1 sparsity pattern of a 3x3 A with fixed distinct values, exact."""
    values = np.arange(1, 10, dtype=np.float64).reshape(3, 3) * np.array([1, -1, 1])
    B = np.array([[1, -2], [3, 5], [-7, 11]], dtype=np.float32)
    for bits in range(512):
        mask = np.array([(bits >> k) & 1 for k in range(9)], dtype=bool).reshape(3, 3)
        A = np.where(mask, values, 0.0)
        rowptr = np.concatenate([[0], np.cumsum(mask.sum(1))]).astype(np.int32)
        colind = np.nonzero(mask)[1].astype(np.int32)
        vals = A[mask].astype(np.float32)
        C, _ = fn(rowptr, colind, vals, B)
        assert np.array_equal(C, A @ B.astype(np.float64)), f"pattern {bits:09b}"


def pin_identity_permutation_scaling(fn):
    rng = np.random.default_rng(7)
    n, N = 37, 5
    B = gen.uniform_b(rng, n, N)
    rp, ci, v = gen.identity_csr(n)
    C, S = fn(rp, ci, v, B)
    assert np.array_equal(C, B.astype(np.float64)), "A = I must give C = B exactly"
    assert np.array_equal(S, np.abs(B.astype(np.float64)))
    perm = rng.permutation(n)
    rp, ci, v = gen.permutation_csr(perm)
    C, _ = fn(rp, ci, v, B)
    assert np.array_equal(C, B[perm].astype(np.float64)), "A = P must give C = P.B exactly"
    for k in (-3, 5):
        rp, ci, v = gen.identity_csr(n, scale=2.0 ** k)
        C, _ = fn(rp, ci, v, B)
        assert np.array_equal(C, B.astype(np.float64) * 2.0 ** k), "A = 2^k I must scale B exactly"


def pin_ones_and_indicator_columns(fn):
    rng = np.random.default_rng(11)
    p = gen.random_csr(rng, 40, 30, 1, mean_row=6, empty_frac=0.2, integer=True)
    A = densify(p.rowptr, p.colind, p.vals, 30)
    ones = np.ones((30, 1), dtype=np.float32)
    C, _ = fn(p.rowptr, p.colind, p.vals, ones)
    assert np.array_equal(C[:, 0], A.sum(axis=1)), "B = ones must give the row sums of A"
    for j in (0, 13, 29):
        e = np.zeros((30, 1), dtype=np.float32)
        e[j, 0] = 1.0
        C, _ = fn(p.rowptr, p.colind, p.vals, e)
        assert np.array_equal(C[:, 0], A[:, j]), f"B = e_{j} must give column {j} of A"


def pin_hand_4x4(fn):
    g = load_golden_hand_4x4()
    C, S = fn(g["rowptr"].astype(np.int32), g["colind"].astype(np.int32),
              g["vals"].astype(np.float32), g["B"].astype(np.float32))
    assert np.array_equal(C, g["C"]), "hand-worked 4x4 C"
    assert np.array_equal(S, g["S"]), "hand-worked 4x4 S"


def pin_double_accumulation(fn):
    """1*2^24 + 1*1 = 16777217 needs more than fp32's 24-bit significand."""
    rowptr = np.array([0, 2], dtype=np.int32)
    colind = np.array([0, 1], dtype=np.int32)
    vals = np.array([1.0, 1.0], dtype=np.float32)
    B = np.array([[2.0 ** 24], [1.0]], dtype=np.float32)
    C, S = fn(rowptr, colind, vals, B)
    assert C[0, 0] == 16777217.0 and S[0, 0] == 16777217.0, "accumulation must be in double"


def pin_integer_exact(fn):
    """Integer data: the result is an int64 matmul, exactly."""
    rng = np.random.default_rng(5)
    p = gen.random_csr(rng, 60, 50, 9, mean_row=10, empty_frac=0.1, duplicates=True, integer=True)
    rows = np.repeat(np.arange(60), np.diff(p.rowptr))
    Ai = np.zeros((60, 50), dtype=np.int64)
    np.add.at(Ai, (rows, p.colind.astype(np.int64)), p.vals.astype(np.int64))
    C, _ = fn(p.rowptr, p.colind, p.vals, p.B)
    assert np.array_equal(C, (Ai @ p.B.astype(np.int64)).astype(np.float64)), "integer SpMM must be exact"


def pin_linearity(fn):
    """C(2 v1 - 3 v2) = 2 C(v1) - 3 C(v2) for integer-valued v1, v2 (all exact)."""
    rng = np.random.default_rng(9)
    p = gen.random_csr(rng, 25, 20, 4, mean_row=5, empty_frac=0.2, integer=True)
    v2 = rng.integers(-4, 5, size=p.nnz).astype(np.float32)
    C1, _ = fn(p.rowptr, p.colind, p.vals, p.B)
    C2, _ = fn(p.rowptr, p.colind, v2, p.B)
    C3, _ = fn(p.rowptr, p.colind, (2 * p.vals - 3 * v2).astype(np.float32), p.B)
    assert np.array_equal(C3, 2 * C1 - 3 * C2), "linearity in vals"


def pin_bf16_decoding(fn):
    """bf16 B must act exactly like torch's bfloat16 -> float32 values of the same bits."""
    rng = np.random.default_rng(13)
    p = gen.random_csr(rng, 30, 24, 16, mean_row=6, empty_frac=0.1, b_dtype="bf16")
    C_bf, S_bf = fn(p.rowptr, p.colind, p.vals, p.B, b_dtype="bf16")
    B32 = _as_f64(p.B, "bf16").astype(np.float32)
    C_f, S_f = fn(p.rowptr, p.colind, p.vals, B32)
    assert np.array_equal(C_bf, C_f) and np.array_equal(S_bf, S_f), "bf16 decoding"
    A = densify(p.rowptr, p.colind, p.vals, 24)
    assert np.all(np.abs(C_bf - A @ _as_f64(p.B, "bf16")) <= 1e-12 * S_bf + 1e-300)


def pin_row_subset(fn):
    rng = np.random.default_rng(17)
    p = gen.random_csr(rng, 30, 20, 6, mean_row=4, empty_frac=0.3)
    C, S = fn(p.rowptr, p.colind, p.vals, p.B)
    rows = np.array([29, 0, 7, 7, 3], dtype=np.int32)
    Cr, Sr = fn(p.rowptr, p.colind, p.vals, p.B, rows=rows)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(Sr, S[rows]), "row subset"


ALL_PINS = [pin_dense_matmul, pin_bruteforce_3x3, pin_identity_permutation_scaling,
            pin_ones_and_indicator_columns, pin_hand_4x4, pin_double_accumulation,
            pin_integer_exact, pin_linearity, pin_bf16_decoding, pin_row_subset]


def oracle_callable(library=None):
    import oracle

    def fn(rowptr, colind, vals, B, b_dtype="f32", rows=None):
        return oracle.spmm_reference(rowptr, colind, vals, B, b_dtype=b_dtype, rows=rows,
                                     library=library)
    return fn


def failing_pins(fn):
    """Names of the pins the given oracle callable fails."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(fn)
        except (AssertionError, ValueError):
            bad.append(pin.__name__)
    return bad
