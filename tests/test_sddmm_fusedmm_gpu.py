"""SDDMM and FusedMM on the GPU vs the CPU oracle, through the C ABI.

Bounds: an SDDMM value is an fp32 dot product, |out - ref| <= 1e-5 * S + 1e-30
with S = sum_n |C_in B_jn|.  FusedMM's values carry that dot-product error into
E, so its bound uses the magnitudes of the whole computation,
S_f[i, n] = sum_j S_ij |D_jn| (the SDDMM bound times |D|), computed with the
oracles."""
import numpy as np
import pytest
import torch

import oracle
from csr_spmm_02_gb300 import gen, spmm
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def problem(seed, M=1200, K=800, N=64, integer=False):
    rng = np.random.default_rng(seed)
    p = gen.random_csr(rng, M, K, N, mean_row=9, empty_frac=0.3, long_rows=[(5, K), (M - 2, 700)])
    if integer:
        C = rng.integers(-2, 3, (M, N)).astype(np.float32)
        B = rng.integers(-2, 3, (K, N)).astype(np.float32)
        D = rng.integers(-2, 3, (K, N)).astype(np.float32)
    else:
        C = rng.uniform(-1, 1, (M, N)).astype(np.float32)
        B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
        D = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    return p, C, B, D


def run_sddmm(p, C, B, T=256, arrays=None, kernel="auto"):
    a = arrays or H.device_arrays(p)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, kernel=kernel, items_per_cta=T)
    out = torch.full((p.nnz,), float("nan"), device="cuda")
    spmm.spmm_csr_sddmm_f32(plan, p.K, a["colind"], torch.from_numpy(C).cuda(), torch.from_numpy(B).cuda(), out)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def run_fusedmm(p, C, B, D, T=256, arrays=None, kernel="auto"):
    a = arrays or H.device_arrays(p)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, kernel=kernel, items_per_cta=T)
    E = torch.full((p.M, p.N), float("nan"), device="cuda")
    spmm.spmm_csr_fusedmm_f32(plan, p.K, a["colind"], torch.from_numpy(C).cuda(), torch.from_numpy(B).cuda(),
                              torch.from_numpy(D).cuda(), E)
    torch.cuda.synchronize()
    assert spmm.spmm_plan_check_device(plan) == 0
    return E.cpu().numpy().astype(np.float64)


def fused_bound(p, C, B, D):
    _, S = oracle.sddmm_reference(p.rowptr, p.colind, C, B)
    Sf, _ = oracle.spmm_reference(p.rowptr, p.colind, S.astype(np.float32), np.abs(D))
    return Sf


@pytest.mark.parametrize("N", [1, 3, 4, 8, 32, 33, 64, 128, 130, 256, 600])
def test_sddmm_parity(N):
    p, C, B, _ = problem(N, N=N)
    got = run_sddmm(p, C, B)
    ref, S = oracle.sddmm_reference(p.rowptr, p.colind, C, B)
    assert np.all(np.abs(got - ref) <= 1e-5 * S + 1e-30)


@pytest.mark.parametrize("N", [4, 8, 12, 16, 20, 32, 60, 64, 100, 128])
def test_sddmm_row_groups(N):
    """Row-class plans with N <= 128 take the group-per-row SDDMM (C row in registers): empty rows,
    rows longer than many rounds, ragged last rounds, lanes past N; integer data is exact."""
    for integer in (False, True):
        p, C, B, _ = problem(300 + N, N=N, integer=integer)
        got = run_sddmm(p, C, B, kernel="row")
        ref, S = oracle.sddmm_reference(p.rowptr, p.colind, C, B)
        if integer:
            assert np.array_equal(got, ref)
        else:
            assert np.all(np.abs(got - ref) <= 1e-5 * S + 1e-30)


@pytest.mark.parametrize("N", [4, 8, 12, 16, 20, 32, 60, 64, 100, 128])
def test_fusedmm_row_groups(N):
    """Row-class plans with N <= 128 take the group-per-row FusedMM (C and E rows in registers)."""
    for integer in (False, True):
        p, C, B, D = problem(400 + N, N=N, integer=integer)
        got = run_fusedmm(p, C, B, D, kernel="row")
        ref, _ = oracle.fusedmm_reference(p.rowptr, p.colind, C, B, D)
        if integer:
            assert np.array_equal(got, ref)
        else:
            H.assert_within(got, ref, fused_bound(p, C, B, D), "f32", f"fusedmm row N={N}")


@pytest.mark.parametrize("N", [1, 3, 4, 8, 32, 33, 64, 128, 130, 256, 600])
def test_fusedmm_parity(N):
    p, C, B, D = problem(100 + N, N=N)
    got = run_fusedmm(p, C, B, D)
    ref, _ = oracle.fusedmm_reference(p.rowptr, p.colind, C, B, D)
    H.assert_within(got, ref, fused_bound(p, C, B, D), "f32", f"fusedmm N={N}")


def band_problem(seed, M, K, below, above, N, integer=False, **kw):
    """A band (test_window_gpu's builder) with dense operands C (M x N), B and D (K x N)."""
    from tests.test_window_gpu import banded
    p = banded(seed, M, K, below, above, N, integer=integer, **kw)
    rng = np.random.default_rng(seed + 7)
    if integer:
        C, D = rng.integers(-2, 3, (M, N)).astype(np.float32), rng.integers(-2, 3, (K, N)).astype(np.float32)
    else:
        C, D = rng.uniform(-1, 1, (M, N)).astype(np.float32), rng.uniform(-1, 1, (K, N)).astype(np.float32)
    return p, C, p.B, D


@pytest.mark.parametrize("kernel", ["window", "window_tc"])
@pytest.mark.parametrize("N", [4, 64, 128, 136, 256, 512])
def test_window_sddmm_fusedmm(kernel, N):
    """Window-class plans: the dense window of each 32-row block from shared memory (a band of
    64 columns spans at most 95 per block), ragged last block, several 128-column passes and a
    partial one (N = 136)."""
    p, C, B, D = band_problem(N, 650, 700, 32, 31, N)
    ref, S = oracle.sddmm_reference(p.rowptr, p.colind, C, B)
    got = run_sddmm(p, C, B, kernel=kernel)
    assert np.all(np.abs(got - ref) <= 1e-5 * S + 1e-30), f"window sddmm N={N}"
    Eref, _ = oracle.fusedmm_reference(p.rowptr, p.colind, C, B, D)
    H.assert_within(run_fusedmm(p, C, B, D, kernel=kernel), Eref, fused_bound(p, C, B, D), "f32",
                    f"window fusedmm N={N}")


@pytest.mark.parametrize("case", ["wide", "duplicates", "unsorted", "empty", "sparse", "long"])
def test_window_sddmm_fusedmm_shapes(case):
    """Blocks that take the gather path (a span over 96 columns, more nonzeros than the staging
    area), duplicate entries (FusedMM counts each occurrence), unsorted columns, empty rows and
    blocks; integer data, so every path must be bitwise exact."""
    kw = {"wide": dict(below=70, above=70), "duplicates": dict(duplicates=True), "unsorted": dict(unsorted=True),
          "empty": dict(empty_every=5), "sparse": dict(sparse_every=3),
          "long": dict(long_rows=[(40, 600), (41, 650), (42, 700), (43, 680)])}[case]
    below, above = kw.pop("below", 32), kw.pop("above", 31)
    for N in (64, 256):
        p, C, B, D = band_problem(90 + N, 400, 720, below, above, N, integer=True, **kw)
        ref, _ = oracle.sddmm_reference(p.rowptr, p.colind, C, B)
        assert np.array_equal(run_sddmm(p, C, B, kernel="window"), ref), f"{case} sddmm N={N}"
        Eref, _ = oracle.fusedmm_reference(p.rowptr, p.colind, C, B, D)
        assert np.array_equal(run_fusedmm(p, C, B, D, kernel="window"), Eref), f"{case} fusedmm N={N}"


def test_window_sddmm_fusedmm_deterministic():
    p, C, B, D = band_problem(3, 500, 520, 32, 31, 256)
    a = H.device_arrays(p)
    assert np.array_equal(run_sddmm(p, C, B, arrays=a, kernel="window"), run_sddmm(p, C, B, arrays=a, kernel="window"))
    assert np.array_equal(run_fusedmm(p, C, B, D, arrays=a, kernel="window"),
                          run_fusedmm(p, C, B, D, arrays=a, kernel="window"))


@pytest.mark.parametrize("N", [8, 64])
def test_integer_exact(N):
    p, C, B, D = problem(200 + N, N=N, integer=True)
    ref, _ = oracle.sddmm_reference(p.rowptr, p.colind, C, B)
    assert np.array_equal(run_sddmm(p, C, B), ref)
    ref, _ = oracle.fusedmm_reference(p.rowptr, p.colind, C, B, D)
    assert np.array_equal(run_fusedmm(p, C, B, D), ref)


def test_deterministic_and_range_sizes():
    p, C, B, D = problem(7, N=32)
    a = H.device_arrays(p)
    e1, e2 = run_fusedmm(p, C, B, D, arrays=a), run_fusedmm(p, C, B, D, arrays=a)
    assert np.array_equal(e1, e2)
    ref, _ = oracle.fusedmm_reference(p.rowptr, p.colind, C, B, D)
    Sf = fused_bound(p, C, B, D)
    for T in (512, 2048, 8192):
        H.assert_within(run_fusedmm(p, C, B, D, T=T, arrays=a), ref, Sf, "f32", f"T={T}")
        out = run_sddmm(p, C, B, T=T, arrays=a)
        sref, S = oracle.sddmm_reference(p.rowptr, p.colind, C, B)
        assert np.all(np.abs(out - sref) <= 1e-5 * S + 1e-30)


def test_scalar_path_misaligned():
    p, C, B, D = problem(9, N=64)
    a = H.device_arrays(p)
    def shifted(x):
        t = torch.from_numpy(x).cuda().reshape(-1)
        buf = torch.empty(t.numel() + 1, device="cuda")
        buf[1:].copy_(t)
        return buf[1:].view(x.shape)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, items_per_cta=256)
    out = torch.empty(p.nnz, device="cuda")
    spmm.spmm_csr_sddmm_f32(plan, p.K, a["colind"], shifted(C), shifted(B), out)
    Ebuf = torch.empty(p.M * p.N + 1, device="cuda")
    E = Ebuf[1:].view(p.M, p.N)
    spmm.spmm_csr_fusedmm_f32(plan, p.K, a["colind"], shifted(C), shifted(B), shifted(D), E)
    torch.cuda.synchronize()
    ref, S = oracle.sddmm_reference(p.rowptr, p.colind, C, B)
    assert np.all(np.abs(out.cpu().numpy() - ref) <= 1e-5 * S + 1e-30)
    Eref, _ = oracle.fusedmm_reference(p.rowptr, p.colind, C, B, D)
    H.assert_within(E, Eref, fused_bound(p, C, B, D), "f32", "fusedmm misaligned")


def test_empty_pattern():
    M, K, N = 50, 20, 16
    p = gen.CsrProblem("empty", M, K, N, np.zeros(M + 1, np.int32), np.zeros(0, np.int32), np.zeros(0, np.float32),
                       np.zeros((K, N), np.float32), "f32")
    a = H.device_arrays(p)
    plan = spmm.spmm_csr_plan(a["rowptr"], M, 0, N)
    E = torch.full((M, N), float("nan"), device="cuda")
    z = torch.zeros((K, N), device="cuda")
    spmm.spmm_csr_fusedmm_f32(plan, K, None, torch.zeros((M, N), device="cuda"), z, z, E)
    torch.cuda.synchronize()
    assert not bool(E.any()) and bool(torch.isfinite(E).all())


@pytest.mark.parametrize("name", ["uniform64k", "banded", "rmat22"])
def test_workload_structures(name):
    """Full-size patterns of three benchmark workloads (N of the workload; banded's bf16 B widened
    exactly to fp32): every SDDMM value and every FusedMM output element against the oracles."""
    p = gen.make_workload(name)
    rng = np.random.default_rng(5)
    C = rng.uniform(-1, 1, (p.M, p.N)).astype(np.float32)
    D = rng.uniform(-1, 1, (p.K, p.N)).astype(np.float32)
    B = p.B if p.b_dtype == "f32" else (p.B.astype(np.uint32) << 16).view(np.float32)
    absD = np.abs(D)
    a = H.device_arrays(p)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N)
    Cd, Bd, Dd = (torch.from_numpy(x).cuda() for x in (C, B, D))
    out = torch.empty(p.nnz, device="cuda")
    spmm.spmm_csr_sddmm_f32(plan, p.K, a["colind"], Cd, Bd, out)
    E = torch.empty((p.M, p.N), device="cuda")
    spmm.spmm_csr_fusedmm_f32(plan, p.K, a["colind"], Cd, Bd, Dd, E)
    torch.cuda.synchronize()
    assert spmm.spmm_plan_check_device(plan) == 0
    out, E = out.cpu().numpy().astype(np.float64), E.cpu().numpy()

    def block(r0, r1):
        rp, ci, _ = H.sub_csr(p, r0, r1)
        ref, S = oracle.sddmm_reference(rp, ci, C[r0:r1], B)
        Eref, _ = oracle.fusedmm_reference(rp, ci, C[r0:r1], B, D)
        Sf, _ = oracle.spmm_reference(rp, ci, S.astype(np.float32), absD)
        return r0, r1, ref, S, Eref, Sf

    for r0, r1, ref, S, Eref, Sf in H.blocks_ahead(block, H.row_blocks(p, 3.0 * p.nnz / p.M * p.N)):
        got = out[int(p.rowptr[r0]):int(p.rowptr[r1])]
        bad = np.abs(got - ref) > 1e-5 * S + 1e-30
        assert not bad.any(), f"{name} sddmm rows {r0}..{r1 - 1}: {int(bad.sum())} values outside the bound"
        H.assert_within(E[r0:r1], Eref, Sf, "f32", f"{name} fusedmm rows {r0}..{r1 - 1}")
