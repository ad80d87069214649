"""Seeded random sweep: many small CSR problems (shapes, densities, skew,
empty rows, duplicates, unsorted columns, both B types, odd N, misaligned B)
through every kernel family, the semirings, SDDMM and FusedMM, each against
the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from csr_spmm_02_gb300 import gen, spmm
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

SEEDS = list(range(48))


def draw(seed):
    rng = np.random.default_rng(10_000 + seed)
    M = int(rng.integers(1, 900))
    K = int(rng.integers(1, 700))
    N = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16, 31, 32, 48, 64, 96, 128, 160, 256, 300]))
    b_dtype = "bf16" if rng.random() < 0.4 else "f32"
    mean = float(rng.choice([0.5, 2, 6, 15, 40]))
    long_rows = [(int(rng.integers(0, M)), int(rng.integers(1, 3 * K + 1)))] if rng.random() < 0.4 else []
    p = gen.random_csr(rng, M, K, N, mean_row=mean, max_row=max(1, 3 * int(mean) + 2),
                       empty_frac=float(rng.choice([0.0, 0.2, 0.6])), long_rows=long_rows,
                       duplicates=bool(rng.random() < 0.3), sort_cols=bool(rng.random() < 0.7), b_dtype=b_dtype)
    misaligned = bool(rng.random() < 0.25)
    return p, misaligned, rng


def device_B(p, misaligned):
    a = H.device_arrays(p)
    if not misaligned:
        return a, a["B"]
    dt = a["B"].dtype
    store = torch.empty(p.K * p.N + 1, dtype=dt, device="cuda")
    B = store[1:].view(p.K, p.N)
    B.copy_(a["B"])
    return a, B


@pytest.mark.parametrize("seed", SEEDS)
def test_fuzz_spmm_all_kernels(seed):
    p, misaligned, _ = draw(seed)
    a, B = device_B(p, misaligned)
    C_ref, S = H.reference(p)
    kernels = ["auto", "row", "balanced", "window", "window_tc", "smalln"]
    for kernel in kernels:
        plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, kernel=kernel, items_per_cta=256)
        C = torch.full((p.M, p.N), float("nan"), device="cuda")
        f = spmm.spmm_csr_f32_exec if p.b_dtype == "f32" else spmm.spmm_csr_bf16f32_exec
        f(plan, p.K, a["colind"], a["vals"], B, C)
        torch.cuda.synchronize()
        assert spmm.spmm_plan_check_device(plan) == 0
        H.assert_within(C, C_ref, S, p.b_dtype, f"seed {seed} {kernel} M={p.M} K={p.K} N={p.N} {p.b_dtype}")
        plan.destroy()


@pytest.mark.parametrize("seed", SEEDS[:24])
def test_fuzz_semiring_sddmm_fusedmm(seed):
    p, misaligned, rng = draw(seed)
    if p.b_dtype == "bf16":  # these operations take fp32 B
        p = gen.CsrProblem(p.name, p.M, p.K, p.N, p.rowptr, p.colind, p.vals,
                           (p.B.astype(np.uint32) << 16).view(np.float32), "f32")
    a, B = device_B(p, misaligned)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, items_per_cta=256)
    add = ["sum", "min", "max"][seed % 3]
    mul = ["mul", "add"][(seed // 3) % 2]
    C = torch.full((p.M, p.N), float("nan"), device="cuda")
    spmm.spmm_csr_semiring_f32_exec(plan, p.K, a["colind"], a["vals"], B, C, add, mul)
    ref, S = oracle.semiring_reference(p.rowptr, p.colind, p.vals, p.B, add, mul)
    torch.cuda.synchronize()
    got = C.cpu().numpy().astype(np.float64)
    if add == "sum":
        H.assert_within(got, ref, S, "f32", f"seed {seed} ({add},{mul})")
    else:
        assert np.array_equal(got, ref.astype(np.float32).astype(np.float64)), f"seed {seed} ({add},{mul})"
    Cd = rng.uniform(-1, 1, (p.M, p.N)).astype(np.float32)
    D = rng.uniform(-1, 1, (p.K, p.N)).astype(np.float32)
    Cg, Dg = torch.from_numpy(Cd).cuda(), torch.from_numpy(D).cuda()
    out = torch.full((max(p.nnz, 1),), float("nan"), device="cuda")[:p.nnz]
    spmm.spmm_csr_sddmm_f32(plan, p.K, a["colind"], Cg, B, out)
    ref_s, S_s = oracle.sddmm_reference(p.rowptr, p.colind, Cd, p.B)
    E = torch.full((p.M, p.N), float("nan"), device="cuda")
    spmm.spmm_csr_fusedmm_f32(plan, p.K, a["colind"], Cg, B, Dg, E)
    ref_f, _ = oracle.fusedmm_reference(p.rowptr, p.colind, Cd, p.B, D)
    Sf, _ = oracle.spmm_reference(p.rowptr, p.colind, S_s.astype(np.float32), np.abs(D))
    torch.cuda.synchronize()
    assert spmm.spmm_plan_check_device(plan) == 0
    if p.nnz:
        H.assert_within(out.cpu().numpy().astype(np.float64), ref_s, S_s, "f32", f"seed {seed} sddmm")
    H.assert_within(E, ref_f, Sf, "f32", f"seed {seed} fusedmm")
