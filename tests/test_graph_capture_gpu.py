"""Exec calls replayed from a CUDA graph.

Once a kernel has run (its first call sets the function's shared-memory
attribute and caches occupancy), an exec call makes no synchronous CUDA call
and allocates nothing, so it can be captured on a stream and replayed.  A
replay reads the captured buffers as they are when it runs: values written
into them before a replay must give what an eager call gives on the same
inputs, bit for bit (every kernel is deterministic), and both must match the
oracle.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from csr_spmm_02_gb300 import gen, spmm
from tests import gpu_helpers as H
from tests.test_window_gpu import banded

pytestmark = pytest.mark.gpu

SPMM_CASES = [("row", "f32", 64), ("balanced", "f32", 32), ("balanced", "bf16", 64), ("smalln", "f32", 4),
              ("window", "f32", 128), ("window_tc", "bf16", 256)]


def _problem(kernel, b_dtype, N, seed):
    if kernel.startswith("window"):
        return banded(seed, 600, 640, 20, 21, N, b_dtype=b_dtype)
    rng = np.random.default_rng(seed)
    return gen.random_csr(rng, 900, 700, N, mean_row=10, empty_frac=0.2, long_rows=[(3, 650)], b_dtype=b_dtype)


@pytest.mark.parametrize("kernel,b_dtype,N", SPMM_CASES)
def test_spmm_exec_replays_from_a_graph(kernel, b_dtype, N):
    p = _problem(kernel, b_dtype, N, 11)
    a = H.device_arrays(p)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, N, kernel=kernel, items_per_cta=256)
    assert plan.info()["kernel"] == kernel
    f = spmm.spmm_csr_f32_exec if b_dtype == "f32" else spmm.spmm_csr_bf16f32_exec
    C_eager = torch.full((p.M, N), float("nan"), device="cuda")
    C_graph = torch.full_like(C_eager, float("nan"))
    f(plan, p.K, a["colind"], a["vals"], a["B"], C_eager)  # first call of this kernel
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        f(plan, p.K, a["colind"], a["vals"], a["B"], C_graph)

    rng = np.random.default_rng(12)
    vals2 = rng.uniform(-1, 1, p.nnz).astype(np.float32)
    Bf = rng.standard_normal((p.K, N)).astype(np.float32)
    B2 = Bf if b_dtype == "f32" else gen.f32_to_bf16_bits(Bf)
    a["vals"].copy_(torch.from_numpy(vals2))
    a["B"].copy_(torch.from_numpy(np.ascontiguousarray(B2.view(np.int16) if b_dtype == "bf16" else B2)))
    g.replay()
    f(plan, p.K, a["colind"], a["vals"], a["B"], C_eager)
    torch.cuda.synchronize()
    assert spmm.spmm_plan_check_device(plan) == 0
    assert torch.equal(C_graph, C_eager), kernel
    C_ref, S = H.reference(dataclasses.replace(p, vals=vals2, B=B2))
    H.assert_within(C_graph, C_ref, S, b_dtype, f"graph replay, {kernel}")
    del g
    plan.destroy()


@pytest.mark.parametrize("kernel", ["balanced", "window"])
def test_sddmm_fusedmm_replay_from_a_graph(kernel):
    N = 64
    p = _problem(kernel, "f32", N, 21)
    a = H.device_arrays(p)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, N, kernel=kernel, items_per_cta=256)
    rng = np.random.default_rng(22)
    Cd = torch.from_numpy(rng.uniform(-1, 1, (p.M, N)).astype(np.float32)).cuda()
    Bd = torch.from_numpy(rng.uniform(-1, 1, (p.K, N)).astype(np.float32)).cuda()
    D = torch.from_numpy(rng.uniform(-1, 1, (p.K, N)).astype(np.float32)).cuda()
    out_e, out_g = torch.empty(p.nnz, device="cuda"), torch.empty(p.nnz, device="cuda")
    E_e, E_g = torch.empty((p.M, N), device="cuda"), torch.empty((p.M, N), device="cuda")
    spmm.spmm_csr_sddmm_f32(plan, p.K, a["colind"], Cd, Bd, out_e)  # first calls of these kernels
    spmm.spmm_csr_fusedmm_f32(plan, p.K, a["colind"], Cd, Bd, D, E_e)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        spmm.spmm_csr_sddmm_f32(plan, p.K, a["colind"], Cd, Bd, out_g)
        spmm.spmm_csr_fusedmm_f32(plan, p.K, a["colind"], Cd, Bd, D, E_g)

    Cn = rng.uniform(-1, 1, (p.M, N)).astype(np.float32)
    Cd.copy_(torch.from_numpy(Cn))
    g.replay()
    spmm.spmm_csr_sddmm_f32(plan, p.K, a["colind"], Cd, Bd, out_e)
    spmm.spmm_csr_fusedmm_f32(plan, p.K, a["colind"], Cd, Bd, D, E_e)
    torch.cuda.synchronize()
    assert spmm.spmm_plan_check_device(plan) == 0
    assert torch.equal(out_g, out_e) and torch.equal(E_g, E_e), kernel
    ref, Sd = oracle.sddmm_reference(p.rowptr, p.colind, Cn, Bd.cpu().numpy())
    got = out_g.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-5 * Sd + 1e-30), f"graph replay sddmm, {kernel}"
    del g
    plan.destroy()
