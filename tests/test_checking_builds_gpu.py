"""The library's checking builds (csr_spmm_02_gb300/build.py, FLAVORS), on the GPU.

bounds (-DSPMM_DEBUG_BOUNDS): every B-row gather and every output store
checks its address against the buffers its launch registered.  The small
parity cases of every kernel family run clean (no access outside its
buffers: the error word stays zero) and match the oracle; a column index
outside [0, K), which the release build leaves undefined, is caught as
SPMM_ERR_OUT_OF_BOUNDS with the access skipped, never a fault.

stage_timeout (-DSPMM_STAGE_SPIN_LIMIT=1): the nnz-balanced kernel's first
wait for its staged copies gives up after one poll, as a bounded wait that
runs out would; the kernel still waits for its copies before it leaves.  The
plan's check and spmm_check_device report SPMM_ERR_DEVICE_TIMEOUT once and
read clear afterwards.
"""
import numpy as np
import pytest
import torch

import oracle
from csr_spmm_02_gb300 import build, gen, spmm
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

OUT_OF_BOUNDS, TIMEOUT = 7, 6


@pytest.fixture(scope="module")
def flavored():
    """Route the binding to a checking build while a test runs."""
    saved = spmm._lib
    libs = {}

    def use(flavor):
        if flavor not in libs:
            libs[flavor] = spmm.load(build.build(flavor=flavor))
        spmm._lib = libs[flavor]
        return libs[flavor]

    yield use
    torch.cuda.synchronize()
    spmm._lib = saved


def banded(rng, M, K, half, N, b_dtype):
    rows = [np.arange(max(0, i - half), min(K, i + half + 1), dtype=np.int32) for i in range(M)]
    rowptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    colind = np.concatenate(rows)
    vals = rng.standard_normal(len(colind)).astype(np.float32)
    Bf = rng.standard_normal((K, N)).astype(np.float32)
    return gen.CsrProblem("band", M, K, N, rowptr, colind, vals, Bf if b_dtype == "f32" else gen.f32_to_bf16_bits(Bf),
                          b_dtype)


def cases(rng):
    skewed = lambda b, N: gen.random_csr(rng, 900, 600, N, mean_row=10, empty_frac=0.3,  # noqa: E731
                                         long_rows=[(5, 600), (890, 300)], b_dtype=b)
    return [("row", skewed("f32", 64)), ("row", skewed("f32", 13)), ("balanced", skewed("f32", 64)),
            ("balanced", skewed("bf16", 64)), ("balanced", skewed("f32", 7)),
            ("window", banded(rng, 300, 320, 20, 128, "f32")), ("window_tc", banded(rng, 300, 320, 20, 256, "bf16")),
            ("smalln", skewed("f32", 4))]


def test_bounds_build_parity_every_family(flavored):
    flavored("bounds")
    rng = np.random.default_rng(71)
    for kernel, p in cases(rng):
        a = H.device_arrays(p)
        C, plan = H.run(p, kernel=kernel, items_per_cta=256, arrays=a)  # asserts a clear error word
        C_ref, S = H.reference(p)
        H.assert_within(C, C_ref, S, p.b_dtype, f"bounds build {kernel}/{p.b_dtype}/N={p.N}")
        if p.b_dtype == "f32":  # SDDMM, FusedMM and a semiring on the same plan
            Cd = rng.uniform(-1, 1, (p.M, p.N)).astype(np.float32)
            D = rng.uniform(-1, 1, (p.K, p.N)).astype(np.float32)
            Cg, Bg, Dg = (torch.from_numpy(x).cuda() for x in (Cd, p.B, D))
            out = torch.empty(p.nnz, device="cuda")
            spmm.spmm_csr_sddmm_f32(plan, p.K, a["colind"], Cg, Bg, out)
            E = torch.empty((p.M, p.N), device="cuda")
            spmm.spmm_csr_fusedmm_f32(plan, p.K, a["colind"], Cg, Bg, Dg, E)
            spmm.spmm_csr_semiring_f32_exec(plan, p.K, a["colind"], a["vals"], a["B"], C, "max", "mul")
            torch.cuda.synchronize()
            assert spmm.spmm_plan_check_device(plan) == 0, f"bounds build {kernel}: SDDMM/FusedMM/semiring"
            ref, Sd = oracle.sddmm_reference(p.rowptr, p.colind, Cd, p.B)
            assert np.all(np.abs(out.cpu().numpy() - ref) <= 1e-5 * Sd + 1e-30)
            Mref, _ = oracle.semiring_reference(p.rowptr, p.colind, p.vals, p.B, "max", "mul")
            assert np.array_equal(C.cpu().numpy().astype(np.float64), Mref.astype(np.float32).astype(np.float64))
        plan.destroy()
    p = cases(rng)[0][1]
    a = H.device_arrays(p)
    for one_call in (spmm.spmm_csr_f32, None):
        C = torch.full((p.M, p.N), float("nan"), device="cuda")
        if one_call:
            one_call(p.M, p.K, p.N, a["rowptr"], a["colind"], a["vals"], a["B"], C)
        else:
            spmm.spmm_csr_f32_noalloc(p.M, p.K, p.N, p.nnz, a["rowptr"], a["colind"], a["vals"], a["B"], C)
        assert spmm.spmm_check_device() == 0
        C_ref, S = H.reference(p)
        H.assert_within(C, C_ref, S, "f32", "bounds build, one-call forms")


@pytest.mark.parametrize("bad", [-3, "K+7"])
def test_bounds_build_catches_a_bad_column(flavored, bad):
    """A column index outside [0, K): every gather it would make is skipped and reported."""
    flavored("bounds")
    rng = np.random.default_rng(5)
    p = gen.random_csr(rng, 700, 400, 32, mean_row=8, empty_frac=0.2, long_rows=[(9, 400)])
    colind = p.colind.copy()
    colind[[3, len(colind) // 2, len(colind) - 1]] = p.K + 7 if bad == "K+7" else bad
    a = H.device_arrays(p)
    a["colind"] = torch.from_numpy(colind).cuda()
    for kernel in ("row", "balanced"):
        plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, kernel=kernel)
        C = torch.empty((p.M, p.N), device="cuda")
        spmm.spmm_csr_f32_exec(plan, p.K, a["colind"], a["vals"], a["B"], C)
        assert spmm.spmm_plan_check_device(plan) == OUT_OF_BOUNDS, kernel
        assert spmm.spmm_plan_check_device(plan) == 0  # read and cleared
        plan.destroy()
    C = torch.empty((p.M, p.N), device="cuda")
    spmm.spmm_csr_f32_noalloc(p.M, p.K, p.N, p.nnz, a["rowptr"], a["colind"], a["vals"], a["B"], C)
    assert spmm.spmm_check_device() == OUT_OF_BOUNDS
    spmm.spmm_csr_f32(p.M, p.K, p.N, a["rowptr"], a["colind"], a["vals"], a["B"], C)
    assert spmm.spmm_check_device() == OUT_OF_BOUNDS
    assert spmm.spmm_check_device() == 0
    # narrow B on a balanced plan: the thread-range kernel (scalar and vector loads)
    for N in (1, 4):
        q = gen.random_csr(rng, 700, 400, N, mean_row=8, empty_frac=0.2, long_rows=[(9, 400)])
        colq = q.colind.copy()
        colq[[3, len(colq) // 2, len(colq) - 1]] = q.K + 7 if bad == "K+7" else bad
        b = H.device_arrays(q)
        b["colind"] = torch.from_numpy(colq).cuda()
        plan = spmm.spmm_csr_plan(b["rowptr"], q.M, q.nnz, N, kernel="balanced")
        C = torch.empty((q.M, N), device="cuda")
        spmm.spmm_csr_f32_exec(plan, q.K, b["colind"], b["vals"], b["B"], C)
        assert spmm.spmm_plan_check_device(plan) == OUT_OF_BOUNDS, f"thread ranges, N={N}"
        assert spmm.spmm_plan_check_device(plan) == 0
        plan.destroy()


def test_stage_timeout_is_reported(flavored):
    """A first wait that gives up is reported by both checks, once."""
    flavored("stage_timeout")
    rng = np.random.default_rng(8)
    p = gen.random_csr(rng, 20000, 5000, 64, mean_row=12, empty_frac=0.3, long_rows=[(77, 5000)])
    a = H.device_arrays(p)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, kernel="balanced", items_per_cta=256)
    assert plan.info()["num_ctas"] > 500
    C = torch.empty((p.M, p.N), device="cuda")
    spmm.spmm_csr_f32_exec(plan, p.K, a["colind"], a["vals"], a["B"], C)
    assert spmm.spmm_plan_check_device(plan) == TIMEOUT
    assert spmm.spmm_plan_check_device(plan) == 0
    plan.destroy()
    # the thread-range kernel (N = 4) takes the same first wait
    q = gen.random_csr(rng, 20000, 5000, 4, mean_row=12, empty_frac=0.3, long_rows=[(77, 5000)])
    b = H.device_arrays(q)
    plan = spmm.spmm_csr_plan(b["rowptr"], q.M, q.nnz, 4, kernel="balanced", items_per_cta=256)
    C4 = torch.empty((q.M, 4), device="cuda")
    spmm.spmm_csr_f32_exec(plan, q.K, b["colind"], b["vals"], b["B"], C4)
    assert spmm.spmm_plan_check_device(plan) == TIMEOUT
    assert spmm.spmm_plan_check_device(plan) == 0
    plan.destroy()
    spmm.spmm_csr_f32_noalloc(p.M, p.K, p.N, p.nnz, a["rowptr"], a["colind"], a["vals"], a["B"], C)
    assert spmm.spmm_check_device() == TIMEOUT
    assert spmm.spmm_check_device() == 0
