"""The row-group kernel for narrow B (N <= 8, r lanes per row) vs the CPU
oracle: every N from 1 to 8, both B types, every group size, the vector and
scalar column paths, integer-exact sums, the planner's choice of r."""
import numpy as np
import pytest
import torch

from csr_spmm_02_gb300 import gen, spmm
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

LANES = [2, 4, 8, 16, 32]


def problem(seed, N, b_dtype="f32", integer=False, M=1700, K=900):
    rng = np.random.default_rng(seed)
    return gen.random_csr(rng, M, K, N, mean_row=14, max_row=60, empty_frac=0.2, b_dtype=b_dtype,
                          integer=integer, duplicates=True, sort_cols=False)


def run(p, lanes=None, B=None, C=None):
    a = H.device_arrays(p)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, kernel="smalln")
    if lanes is not None:
        spmm.spmm_plan_set_group_lanes(plan, lanes)
    if C is None:
        C = torch.full((p.M, p.N), float("nan"), device="cuda")
    f = spmm.spmm_csr_f32_exec if p.b_dtype == "f32" else spmm.spmm_csr_bf16f32_exec
    f(plan, p.K, a["colind"], a["vals"], a["B"] if B is None else B, C)
    torch.cuda.synchronize()
    return C, plan


@pytest.mark.parametrize("b_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("lanes", LANES)
def test_parity(b_dtype, N, lanes):
    p = problem(10 * N + lanes, N, b_dtype)
    C, _ = run(p, lanes)
    C_ref, S = H.reference(p)
    H.assert_within(C, C_ref, S, b_dtype, f"smalln/{b_dtype}/N={N}/r={lanes}")


@pytest.mark.parametrize("N", [4, 8])
@pytest.mark.parametrize("lanes", [2, 8, 32])
def test_integer_exact(N, lanes):
    p = problem(N + lanes, N, integer=True)
    C, _ = run(p, lanes)
    C_ref, _ = H.reference(p)
    H.assert_exact(C, C_ref, f"N={N}/r={lanes}")


@pytest.mark.parametrize("N", [4, 8])
def test_misaligned_uses_scalar_columns(N):
    p = problem(3, N)
    Bs = torch.empty(p.K * p.N + 1, device="cuda")
    B = Bs[1:].view(p.K, p.N)
    B.copy_(torch.from_numpy(p.B))
    C, _ = run(p, 8, B=B)
    C_ref, S = H.reference(p)
    H.assert_within(C, C_ref, S, "f32", f"misaligned N={N}")


def test_planner_and_setter():
    rng = np.random.default_rng(4)
    for mean, expect in ((3, 2), (12, 4), (30, 8), (60, 16), (200, 32)):
        p = gen.random_csr(rng, 400, 2000, 4, mean_row=mean, max_row=2 * mean, empty_frac=0.0)
        a = H.device_arrays(p)
        plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, 4)
        info = plan.info()
        assert info["kernel"] == "smalln", info
        m = p.nnz / p.M
        r = 2
        while r < 32 and 4 * r < m:
            r *= 2
        assert info["group_lanes"] == r
    with pytest.raises(spmm.SpmmError):
        spmm.spmm_plan_set_group_lanes(plan, 3)
    wide = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, 64)
    with pytest.raises(spmm.SpmmError):
        spmm.spmm_plan_set_group_lanes(wide, 8)


def test_empty_rows_and_tail():
    p = problem(5, 4, M=32 * 7 + 3)
    p.rowptr[:] = np.minimum(p.rowptr, p.rowptr[100])  # rows 100.. empty
    p = gen.CsrProblem("t", p.M, p.K, p.N, p.rowptr, p.colind[:p.rowptr[-1]], p.vals[:p.rowptr[-1]], p.B, "f32")
    C, _ = run(p, 16)
    C_ref, S = H.reference(p)
    H.assert_within(C, C_ref, S, "f32", "empty tail")
    assert not bool(C[100:].any())
