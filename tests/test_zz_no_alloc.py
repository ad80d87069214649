"""The allocation-free entry point, spmm_csr_f32_noalloc.

It is for callers that must not allocate device memory while they multiply
(an arena that owns all memory, a real-time loop, an embedder's allocator):
its scratch lives in a fixed array inside the library.  The GPU test calls it
twice in a row through the C ABI, on two different problems, and compares each
result with the ordinary one-call entry point spmm_csr_f32 within the fp32
acceptance bound the other parity tests use.  This file is named to be
collected last and needs no state from other tests.
"""
import ctypes

import numpy as np
import pytest

import __graft_entry__
from csr_spmm_02_gb300 import gen, spmm
from tests import gpu_helpers as H


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return spmm.load()


def test_noalloc_rejects_before_any_cuda_call(lib):
    null = ctypes.c_void_p()
    f = lib.spmm_csr_f32_noalloc
    assert f(-1, 4, 4, 0, null, null, null, null, null, null) == 1  # INVALID_ARG
    assert f(0, 4, 4, 0, null, null, null, null, null, null) == 0  # M = 0: nothing to do
    assert f(4, 4, 4, 0, null, null, null, null, null, null) == 1  # NULL rowptr
    big = ctypes.c_void_p(256)
    # 10^8 rows + 10^9 nonzeros at N = 64 needs far more than the fixed scratch: UNSUPPORTED
    assert f(100_000_000, 4, 64, 1_000_000_000, big, big, big, big, big, null) == 3


@pytest.mark.gpu
def test_noalloc_matches_one_call_twice(lib):
    import torch
    rng = np.random.default_rng(31)
    problems = [
        gen.random_csr(rng, 3000, 2000, 64, mean_row=12, empty_frac=0.4, long_rows=[(10, 2000), (2990, 1500)]),
        gen.random_csr(rng, 1700, 900, 32, mean_row=6, empty_frac=0.2, long_rows=[(0, 900)]),
    ]
    for p in problems:  # two calls in a row, different shapes
        a = H.device_arrays(p)
        C_ref = torch.full((p.M, p.N), float("nan"), device="cuda")
        spmm.spmm_csr_f32(p.M, p.K, p.N, a["rowptr"], a["colind"], a["vals"], a["B"], C_ref)
        C_new = torch.full((p.M, p.N), float("nan"), device="cuda")
        spmm.spmm_csr_f32_noalloc(p.M, p.K, p.N, p.nnz, a["rowptr"], a["colind"], a["vals"], a["B"], C_new)
        torch.cuda.synchronize()
        _, S = H.reference(p)
        H.assert_within(C_new, C_ref.cpu().numpy().astype(np.float64), S, "f32", "noalloc vs one-call")
