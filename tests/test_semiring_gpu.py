"""Semiring SpMM on the GPU vs the CPU oracle, through the C ABI.

min and max are exact in any order, so the GPU result must equal the
oracle's value rounded to binary32, bit for bit (+-inf for empty rows);
sums are held to the SpMM bound |C - ref| <= 1e-5 * S + 1e-30."""
import numpy as np
import pytest
import torch

import oracle
from csr_spmm_02_gb300 import gen, spmm
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

OPS = [(a, m) for a in ("sum", "min", "max") for m in ("mul", "add")]


def run(p, add, mul, T=256, kernel="auto", B=None, C=None):
    a = H.device_arrays(p)
    Bd = a["B"] if B is None else B
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, kernel=kernel, items_per_cta=T)
    if C is None:
        C = torch.full((p.M, p.N), float("nan"), device="cuda")
    spmm.spmm_csr_semiring_f32_exec(plan, p.K, a["colind"], a["vals"], Bd, C, add, mul)
    torch.cuda.synchronize()
    assert spmm.spmm_plan_check_device(plan) == 0
    return C


def check(C, p, add, mul, what=""):
    ref, S = oracle.semiring_reference(p.rowptr, p.colind, p.vals, p.B, add, mul)
    got = C.cpu().numpy().astype(np.float64)
    if add == "sum":
        H.assert_within(got, ref, S, "f32", f"{add}/{mul} {what}")
    else:
        expect = ref.astype(np.float32).astype(np.float64)
        bad = got != expect
        assert not bad.any(), f"{add}/{mul} {what}: {int(bad.sum())} elements differ, first {np.argwhere(bad)[0]}"


def problem(seed, M=1300, K=700, N=8, integer=False):
    rng = np.random.default_rng(seed)
    return gen.random_csr(rng, M, K, N, mean_row=9, empty_frac=0.3, long_rows=[(4, K), (M - 2, 650)],
                          duplicates=True, sort_cols=False, integer=integer)


@pytest.mark.parametrize("add,mul", OPS)
@pytest.mark.parametrize("N", [1, 3, 4, 8, 33, 64, 128])
def test_semiring_parity(add, mul, N):
    p = problem(N, N=N)
    check(run(p, add, mul), p, add, mul, f"N={N}")


@pytest.mark.parametrize("add,mul", OPS)
@pytest.mark.parametrize("T", [512, 2048, 8192])
def test_range_sizes_and_kernels(add, mul, T):
    p = problem(T, N=16)
    for kernel in ("auto", "balanced"):
        check(run(p, add, mul, T=T, kernel=kernel), p, add, mul, f"T={T}/{kernel}")


@pytest.mark.parametrize("add,mul", OPS)
def test_misaligned_scalar_path(add, mul):
    p = problem(5, N=12)
    a = H.device_arrays(p)
    Bs = torch.empty(p.K * p.N + 1, device="cuda")
    B = Bs[1:].view(p.K, p.N)
    B.copy_(a["B"])
    check(run(p, add, mul, B=B), p, add, mul, "misaligned")


def test_integer_sum_exact():
    p = problem(6, N=8, integer=True)
    for mul in ("mul", "add"):
        C = run(p, "sum", mul)
        ref, _ = oracle.semiring_reference(p.rowptr, p.colind, p.vals, p.B, "sum", mul)
        assert np.array_equal(C.cpu().numpy().astype(np.float64), ref), mul


def test_empty_matrix_gives_identity():
    M, K, N = 50, 20, 4
    p = gen.CsrProblem("empty", M, K, N, np.zeros(M + 1, np.int32), np.zeros(0, np.int32),
                       np.zeros(0, np.float32), np.ones((K, N), np.float32), "f32")
    for add, ident in (("sum", 0.0), ("min", np.inf), ("max", -np.inf)):
        C = run(p, add, "add")
        assert bool((C == ident).all()), add


def test_deterministic():
    p = problem(7, N=32)
    for add, mul in (("sum", "mul"), ("sum", "add"), ("min", "add")):
        assert torch.equal(run(p, add, mul), run(p, add, mul))


def test_shortest_paths_on_rmat_pattern():
    """Iterating x <- min(x, A (min,+) x) on the GPU reaches scipy's Dijkstra
    distances on a scale-16 R-MAT graph with integer weights (exact)."""
    import scipy.sparse as sp
    from scipy.sparse.csgraph import dijkstra
    rowptr, colind = gen.rmat_structure(np.random.default_rng(8), 16, 8)
    n = len(rowptr) - 1
    w = np.random.default_rng(9).integers(1, 16, len(colind)).astype(np.float32)
    # row i holds the edges j -> i: (A (min,+) x)[i] = min_j w + x[j]
    rp = torch.from_numpy(rowptr).cuda()
    ci = torch.from_numpy(colind).cuda()
    wv = torch.from_numpy(w).cuda()
    plan = spmm.spmm_csr_plan(rp, n, len(colind), 1)
    x = torch.full((n, 1), float("inf"), device="cuda")
    x[0, 0] = 0.0
    y = torch.empty_like(x)
    for _ in range(200):
        spmm.spmm_csr_semiring_f32_exec(plan, n, ci, wv, x, y, "min", "add")
        nx = torch.minimum(x, y)
        if torch.equal(nx, x):
            break
        x = nx
    rows = np.repeat(np.arange(n), np.diff(rowptr))
    G = sp.csr_matrix((w.astype(np.float64), (colind, rows)), shape=(n, n))  # edge j -> i
    G.sum_duplicates()
    ref = dijkstra(G, directed=True, indices=0)
    assert np.array_equal(x[:, 0].cpu().numpy().astype(np.float64), ref)
