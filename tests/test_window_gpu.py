"""The window kernels vs the CPU oracle.  CUDA-core window (B rows staged per
CTA, reused across 4 rows per warp): both of its paths (window and gather),
the boundary between them, duplicates and unsorted columns, CTAs too large
to stage, empty CTAs, several column tiles, determinism.  Tensor-core window
(bf16 B, 128-row tiles, tcgen05): spans of one to four 64-column chunks and
beyond (gather path), N from 16 to 256, ragged M, K inside the last chunk,
duplicates and unsorted rows (gather path), exact integer products."""
import numpy as np
import pytest
import torch

from csr_spmm_02_gb300 import gen
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

ROWS_PER_CTA = 32
WINDOW_ROWS = 128  # B rows the shared-memory window holds for 512-byte tile rows


def banded(seed, M, K, below, above, N, b_dtype="f32", integer=False, duplicates=False, unsorted=False,
           empty_every=0, sparse_every=0, long_rows=(), ends_only=False):
    """Row i holds columns max(0, i-below) .. min(K-1, i+above) (with ends_only,
    only the two ends and the diagonal of that range), with options."""
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(M):
        if (empty_every and i % empty_every == 3) or (sparse_every and i % sparse_every):
            rows.append(np.zeros(0, np.int32))
            continue
        if i in dict(long_rows):
            cols = np.sort(rng.choice(K, dict(long_rows)[i], replace=False)).astype(np.int32)
        else:
            cols = np.arange(max(0, i - below), min(K - 1, i + above) + 1, dtype=np.int32)
            if ends_only:
                cols = np.unique(np.array([cols[0], min(i, K - 1), cols[-1]], np.int32))
        if duplicates and len(cols) and i % 5 == 0:
            cols = np.concatenate([cols, cols[:2]])
        if unsorted:
            cols = rng.permutation(cols).astype(np.int32)
        rows.append(cols)
    rowptr = np.zeros(M + 1, np.int64)
    rowptr[1:] = np.cumsum([len(r) for r in rows])
    colind = np.concatenate(rows).astype(np.int32) if rowptr[-1] else np.zeros(0, np.int32)
    nnz = int(rowptr[-1])
    if integer:
        vals = rng.integers(-2, 3, nnz).astype(np.float32)
        Bf = rng.integers(-3, 4, (K, N)).astype(np.float32)
    else:
        vals = rng.standard_normal(nnz).astype(np.float32)
        Bf = rng.standard_normal((K, N)).astype(np.float32)
    B = Bf if b_dtype == "f32" else gen.f32_to_bf16_bits(Bf)
    return gen.CsrProblem("banded-test", M, K, N, rowptr.astype(np.int32), colind, vals, B, b_dtype)


def check(p, kernel="window"):
    C, plan = H.run(p, kernel=kernel)
    info = plan.info()
    C_ref, S = H.reference(p)
    H.assert_within(C, C_ref, S, p.b_dtype, f"{kernel}/{p.b_dtype}/N={p.N}")
    plan.destroy()
    return C, info


@pytest.mark.parametrize("b_dtype,N", [("f32", 128), ("f32", 136), ("f32", 256), ("f32", 260),
                                       ("bf16", 256), ("bf16", 264), ("bf16", 512)])
def test_banded_parity(b_dtype, N):
    p = banded(N, 1000, 1000, 32, 31, N, b_dtype=b_dtype)
    _, info = check(p, kernel="auto")
    assert info["kernel"] == "window_tc"  # bf16 runs on the tensor cores, fp32 on the CUDA-core window


@pytest.mark.parametrize("width", [95, 96, 97])  # CTA spans of 127, 128 and 129 B rows
def test_span_boundary(width):
    below = width // 2
    p = banded(width, 700, 800, below, width - below, 128, ends_only=True)
    check(p)


@pytest.mark.parametrize("b_dtype", ["f32", "bf16"])
def test_integer_duplicates_unsorted_exact(b_dtype):
    p = banded(7, 900, 950, 20, 25, 256, b_dtype=b_dtype, integer=True, duplicates=True, unsorted=True,
               empty_every=7)
    C, _ = H.run(p, kernel="window")
    C_ref, _ = H.reference(p)
    H.assert_exact(C, C_ref, f"window/{b_dtype}")


def test_long_rows_use_the_gather_path():
    # a CTA holding a 3000-nonzero row cannot stage; its neighbours still use the window
    p = banded(8, 640, 4000, 10, 10, 128, long_rows=((40, 3000), (300, 1500), (601, 2100)))
    check(p)


def test_empty_ctas_and_ragged_tail():
    p = banded(9, 32 * 9 + 7, 300, 3, 3, 256, b_dtype="bf16", sparse_every=100)  # CTAs 1, 2, 4, 5, 7 empty
    C, _ = check(p)
    rp = p.rowptr
    empty = np.flatnonzero(np.diff(rp) == 0)
    assert not bool(C[torch.from_numpy(empty).cuda()].any())
    q = banded(10, 32 * 3 + 1, 64, 0, 0, 128)  # one diagonal, last CTA has one row
    check(q)
    z = gen.CsrProblem("empty", 70, 50, 128, np.zeros(71, np.int32), np.zeros(0, np.int32),
                       np.zeros(0, np.float32), np.ones((50, 128), np.float32), "f32")
    C, _ = H.run(z, kernel="window")
    assert not bool(C.any())


def test_scattered_columns_use_the_gather_path():
    rng = np.random.default_rng(11)
    for N, b in ((128, "f32"), (256, "bf16")):
        p = gen.random_csr(rng, 1200, 5000, N, mean_row=12, empty_frac=0.2, long_rows=[(17, 2500)], b_dtype=b)
        check(p)


def test_deterministic():
    p = banded(12, 2000, 2000, 32, 31, 256, b_dtype="bf16")
    C1, _ = H.run(p, kernel="window")
    C2, _ = H.run(p, kernel="window")
    assert torch.equal(C1, C2)


# ---- tensor-core window ----------------------------------------------------

@pytest.mark.parametrize("N", [16, 32, 48, 128, 256])
def test_tc_banded_parity(N):
    p = banded(N + 500, 1000, 1000, 32, 31, N, b_dtype="bf16")
    _, info = check(p, kernel="window_tc")
    assert info["kernel"] == "window_tc"


@pytest.mark.parametrize("below,above", [(0, 0), (10, 20), (60, 3), (32, 32), (33, 32), (100, 90), (150, 150)])
def test_tc_spans_and_gather_fallback(below, above):
    # 128-row tiles span 128 + below + above columns: 2 or 3 chunks up to 192 columns (32, 32), then the
    # gather path (33, 32 and wider)
    p = banded(below + above, 777, 900, below, above, 64, b_dtype="bf16")
    check(p, kernel="window_tc")


@pytest.mark.parametrize("N", [16, 256])
def test_tc_integer_exact(N):
    p = banded(N + 1, 700, 740, 40, 21, N, b_dtype="bf16", integer=True, empty_every=9)
    C, _ = H.run(p, kernel="window_tc")
    C_ref, _ = H.reference(p)
    H.assert_exact(C, C_ref, f"window_tc/N={N}")


def test_tc_small_k_and_ragged_tail():
    p = banded(3, 200, 70, 16, 16, 32, b_dtype="bf16")  # K = 70: the window ends inside a chunk
    check(p, kernel="window_tc")
    q = banded(4, 129, 129, 5, 5, 16, b_dtype="bf16")  # last tile holds one row
    check(q, kernel="window_tc")


def test_tc_duplicates_and_unsorted_use_gather():
    p = banded(5, 600, 600, 8, 8, 64, b_dtype="bf16", integer=True, duplicates=True)
    C, _ = H.run(p, kernel="window_tc")
    H.assert_exact(C, H.reference(p)[0], "duplicates")
    q = banded(6, 600, 600, 8, 8, 64, b_dtype="bf16", integer=True, unsorted=True)
    C, _ = H.run(q, kernel="window_tc")
    H.assert_exact(C, H.reference(q)[0], "unsorted")


def test_tc_empty_tiles_and_fp32_fallback():
    p = banded(7, 128 * 5 + 3, 300, 3, 3, 256, b_dtype="bf16", sparse_every=200)  # tiles 1, 3 empty
    C, _ = check(p, kernel="window_tc")
    empty = np.flatnonzero(np.diff(p.rowptr) == 0)
    assert not bool(C[torch.from_numpy(empty).cuda()].any())
    q = banded(8, 500, 500, 20, 20, 128)  # fp32 B: the CUDA-core window kernel runs
    check(q, kernel="window_tc")


def test_tc_deterministic():
    p = banded(9, 2000, 2000, 32, 31, 256, b_dtype="bf16")
    C1, _ = H.run(p, kernel="window_tc")
    C2, _ = H.run(p, kernel="window_tc")
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("scale_exp", [-100, -112, -120, -128, -135, -140])
def test_tc_window_tiny_values(scale_exp):
    """Rows whose values all lie near 2^scale_exp, next to ordinary rows, on the
    tensor-core window path.  The three-term bf16 split is exact only for
    |v| >= 2^-110 (at 2^-128 the hi term is a bf16 subnormal, at 2^-135 and
    below it rounds to zero), so tiles holding smaller values must take the
    fp32 gather path; every element must meet the bf16-B bound 8e-3 * S.
    (Values much below 2^-140 would put exact results in the fp32 subnormal
    range, where no fp32 output can meet a purely relative bound.)"""
    p = banded(5, 650, 650, 32, 31, 128, b_dtype="bf16")
    rng = np.random.default_rng(200 - scale_exp)
    tiny_rows = [0, 1, 130, 131, 300, 645]  # rows of several 128-row tiles, incl. the ragged last one
    for r in tiny_rows:
        a, b = int(p.rowptr[r]), int(p.rowptr[r + 1])
        assert b > a
        mant = rng.uniform(1.0, 2.0, b - a) * rng.choice([-1.0, 1.0], b - a)
        p.vals[a:b] = (mant * 2.0 ** scale_exp).astype(np.float32)
    _, info = check(p, kernel="auto")
    assert info["kernel"] == "window_tc"
