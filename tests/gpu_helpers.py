"""Helpers for the GPU parity tests: move a CsrProblem to the device, run the
CUDA path through the C ABI, compare with the CPU oracle."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from csr_spmm_02_gb300 import spmm

# Acceptance bounds per element: |C_gpu - C_oracle| <= REL * S + ABS, where S
# is the oracle's sum of |vals[p] * B[colind[p], n]|.
TOL = {"f32": (1e-5, 1e-30), "bf16": (8e-3, 0.0)}


def device_arrays(p, dev="cuda"):
    B = p.B.view(np.int16) if p.b_dtype == "bf16" else p.B
    return dict(rowptr=torch.from_numpy(p.rowptr).to(dev), colind=torch.from_numpy(p.colind).to(dev),
                vals=torch.from_numpy(p.vals).to(dev), B=torch.from_numpy(np.ascontiguousarray(B)).to(dev))


def run(p, kernel="auto", items_per_cta=0, arrays=None, C=None, plan=None, stream=None):
    """C = A . B on the GPU via a plan; returns (C tensor, plan)."""
    a = arrays or device_arrays(p)
    if C is None:
        C = torch.full((p.M, p.N), float("nan"), device="cuda")
    if plan is None:
        plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, kernel=kernel, items_per_cta=items_per_cta,
                                  stream=stream)
    f = spmm.spmm_csr_f32_exec if p.b_dtype == "f32" else spmm.spmm_csr_bf16f32_exec
    f(plan, p.K, a["colind"], a["vals"], a["B"], C, stream=stream)
    torch.cuda.synchronize()
    assert spmm.spmm_plan_check_device(plan) == 0, "device error word set"
    return C, plan


def reference(p, rows=None):
    return oracle.spmm_reference(p.rowptr, p.colind, p.vals, p.B, b_dtype=p.b_dtype, rows=rows)


def oracle_threads():
    return max(1, min(32, os.cpu_count() or 1))


def row_blocks(p, per_row_work=None):
    """Consecutive row blocks [r0, r1) covering all M rows, each ~2e6 multiply-adds."""
    per_row = per_row_work or max(1.0, float(p.nnz) / max(1, p.M)) * p.N
    block_rows = int(max(256, min(p.M, 2e6 / per_row)))
    return [(r0, min(p.M, r0 + block_rows)) for r0 in range(0, p.M, block_rows)]


def blocks_ahead(fn, blocks):
    """Yield fn(r0, r1) for each block in order, computed on the host's cores
    (a thread pool; the oracle's ctypes calls release the GIL) a few blocks
    ahead of the consumer, so a full-size output is checked element by
    element without holding its whole float64 reference."""
    import concurrent.futures as cf
    nthreads = oracle_threads()
    with cf.ThreadPoolExecutor(nthreads) as ex:
        ahead = 2 * nthreads
        futs = [ex.submit(fn, *b) for b in blocks[:ahead]]
        nxt = ahead
        while futs:
            yield futs.pop(0).result()
            if nxt < len(blocks):
                futs.append(ex.submit(fn, *blocks[nxt]))
                nxt += 1


def sub_csr(p, r0, r1):
    """(rowptr, colind, vals) of rows r0..r1-1, rowptr rebased to 0."""
    a, b = int(p.rowptr[r0]), int(p.rowptr[r1])
    return (p.rowptr[r0:r1 + 1] - p.rowptr[r0]).astype(np.int32), p.colind[a:b], p.vals[a:b]


def reference_blocks(p):
    """Yield (r0, r1, C_ref, S) for consecutive row blocks covering all M rows."""
    def one(r0, r1):
        C, S = reference(p, rows=np.arange(r0, r1, dtype=np.int32))
        return r0, r1, C, S
    yield from blocks_ahead(one, row_blocks(p))


def assert_within_all(C_host, p, what=""):
    """Every element of C_host (M x N, on the host) against the oracle's bound."""
    for r0, r1, C_ref, S in reference_blocks(p):
        assert_within(C_host[r0:r1], C_ref, S, p.b_dtype, f"{what} rows {r0}..{r1 - 1}")


def assert_within(C_gpu, C_ref, S, b_dtype, what=""):
    got = C_gpu.detach().cpu().numpy().astype(np.float64) if isinstance(C_gpu, torch.Tensor) else C_gpu
    rel, absf = TOL[b_dtype]
    assert got.shape == C_ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - C_ref)
    bound = rel * S + absf
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside |d| <= {rel}*S + {absf}; "
                             f"first at {tuple(i)}: got {got[tuple(i)]!r} ref {C_ref[tuple(i)]!r} S {S[tuple(i)]!r}")


def assert_exact(C_gpu, C_ref, what=""):
    got = C_gpu.detach().cpu().numpy().astype(np.float64)
    assert np.array_equal(got, C_ref), f"{what}: not bitwise equal to the exact result"
