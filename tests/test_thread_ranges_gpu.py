"""The thread-range kernel: balanced plans with N <= 2 (fp32 or bf16 B, scalar
loads), N = 4 (16-byte aligned fp32 B) and N = 8 (16-byte aligned bf16 B), one
thread per slice of each merge-path range.

Range sizes of 256, 2048 and 8192 items (1, 8 and 32 items per thread), rows
that end inside a thread, rows that cross threads, warps and ranges (long
rows over many CTAs), empty rows and duplicates.  Small integers make every
partial sum exact in fp32, so the result must equal the oracle's bit for bit
whatever the summation order.  The neighbouring widths (N = 3, misaligned
N = 4 and bf16 N = 8, fp32 N = 8), which stay on the lane-group kernel, are
checked beside them.
"""
import numpy as np
import pytest
import torch

from csr_spmm_02_gb300 import gen, spmm
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _problem(seed, N, b_dtype, integer, M=3000, K=900):
    rng = np.random.default_rng(seed)
    return gen.random_csr(rng, M, K, N, mean_row=6, empty_frac=0.3, duplicates=True, b_dtype=b_dtype,
                          integer=integer, long_rows=[(7, K), (M // 2, 700), (M - 1, 850)])


SHAPES = [(1, "f32"), (2, "f32"), (4, "f32"), (1, "bf16"), (2, "bf16"), (3, "f32"), (8, "f32"), (8, "bf16")]


@pytest.mark.parametrize("T", [256, 2048, 8192])
@pytest.mark.parametrize("N,b_dtype", SHAPES)
def test_exact_integers(N, b_dtype, T):
    p = _problem(10 * N + T, N, b_dtype, integer=True)
    C, plan = H.run(p, kernel="balanced", items_per_cta=T)
    assert plan.info()["kernel"] == "balanced"
    C_ref, _ = H.reference(p)
    H.assert_exact(C, C_ref, f"N={N} {b_dtype} T={T}")
    plan.destroy()


@pytest.mark.parametrize("N,b_dtype", [(1, "f32"), (2, "bf16"), (4, "f32"), (8, "bf16")])
def test_random_values_within_bound(N, b_dtype):
    p = _problem(500 + N, N, b_dtype, integer=False)
    C, plan = H.run(p, kernel="balanced", items_per_cta=2048)
    C_ref, S = H.reference(p)
    H.assert_within(C, C_ref, S, b_dtype, f"N={N} {b_dtype}")
    plan.destroy()


@pytest.mark.parametrize("N,b_dtype", [(2, "f32"), (4, "f32"), (8, "bf16")])
def test_misaligned_b(N, b_dtype):
    p = _problem(700 + N, N, b_dtype, integer=True)
    a = H.device_arrays(p)
    flat = torch.empty(p.K * N + 1, dtype=a["B"].dtype, device="cuda")
    flat[1:] = a["B"].reshape(-1)
    a["B"] = flat[1:]  # one element past a 16-byte boundary
    C, plan = H.run(p, kernel="balanced", items_per_cta=512, arrays=a)
    C_ref, _ = H.reference(p)
    H.assert_exact(C, C_ref, f"misaligned B, N={N}")
    plan.destroy()


@pytest.mark.parametrize("N", [1, 4])
def test_one_long_row_and_empty_rows(N):
    """A row of 60,000 nonzeros between runs of empty rows: the row crosses
    every thread of about 30 ranges (slot 0 of each, slot 1 of the first)."""
    rng = np.random.default_rng(9)
    M, K = 4000, 5000
    lens = np.zeros(M, np.int64)
    lens[1000] = 60000
    lens[rng.integers(0, M, 300)] += rng.integers(1, 5, 300)
    rowptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    nnz = int(rowptr[-1])
    colind = rng.integers(0, K, nnz).astype(np.int32)
    vals = rng.integers(-2, 3, nnz).astype(np.float32)
    B = rng.integers(-3, 4, (K, N)).astype(np.float32)
    p = gen.CsrProblem("one-long-row", M, K, N, rowptr, colind, vals, B, "f32")
    for T in (256, 2048):
        C, plan = H.run(p, kernel="balanced", items_per_cta=T)
        C_ref, _ = H.reference(p)
        H.assert_exact(C, C_ref, f"one long row, T={T}")
        plan.destroy()


def test_deterministic():
    p = _problem(77, 4, "f32", integer=False)
    a = H.device_arrays(p)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, kernel="balanced", items_per_cta=2048)
    outs = []
    for _ in range(3):
        C = torch.full((p.M, p.N), float("nan"), device="cuda")
        spmm.spmm_csr_f32_exec(plan, p.K, a["colind"], a["vals"], a["B"], C)
        outs.append(C)
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    plan.destroy()


@pytest.mark.parametrize("N", [1, 3, 4, 8])
def test_default_ranges_for_sddmm_and_fusedmm(N):
    """Plans at N = 1, 3, 4 and 8 take 3840-item ranges by default; the merge-path
    SDDMM and fused kernels run on the same ranges."""
    import oracle
    p = _problem(900 + N, N, "f32", integer=True)
    a = H.device_arrays(p)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, N, kernel="balanced")
    assert plan.info()["items_per_cta"] == 3840
    rng = np.random.default_rng(N)
    Cd = rng.integers(-2, 3, (p.M, N)).astype(np.float32)
    Bd = rng.integers(-2, 3, (p.K, N)).astype(np.float32)
    D = rng.integers(-2, 3, (p.K, N)).astype(np.float32)
    Cg, Bg, Dg = (torch.from_numpy(x).cuda() for x in (Cd, Bd, D))
    out = torch.empty(p.nnz, device="cuda")
    spmm.spmm_csr_sddmm_f32(plan, p.K, a["colind"], Cg, Bg, out)
    E = torch.empty((p.M, N), device="cuda")
    spmm.spmm_csr_fusedmm_f32(plan, p.K, a["colind"], Cg, Bg, Dg, E)
    torch.cuda.synchronize()
    assert spmm.spmm_plan_check_device(plan) == 0
    ref, _ = oracle.sddmm_reference(p.rowptr, p.colind, Cd, Bd)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), ref)
    Eref, _ = oracle.fusedmm_reference(p.rowptr, p.colind, Cd, Bd, D)
    assert np.array_equal(E.cpu().numpy().astype(np.float64), Eref)
    plan.destroy()
