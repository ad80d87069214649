"""The allocation-free entry point, spmm_csr_f32_noalloc, and the one-call
forms' error word (spmm_check_device).

spmm_csr_f32_noalloc is for callers that must not allocate device memory
while they multiply (an arena or pool that owns all memory, a real-time loop
that cannot take an allocation's synchronisation or failure, an embedder
whose allocator must not be bypassed): its scratch lives in a fixed array
inside the library.  The GPU tests call it through the C ABI and check every
output element against the CPU oracle within the fp32 acceptance bound the
other parity tests use, and against the ordinary one-call entry point
spmm_csr_f32 on two calls in a row.  Cases: the vector path and the scalar
path (N % 4 != 0), a misaligned B, a row of 100,000 nonzeros, a second call
with more ranges than the first (no stale carry rows), a problem whose
scratch just fits the array, and an nnz that differs from rowptr[M] (the
device check leaves C unwritten and spmm_check_device reports it).  The
file is named to be collected last and needs no state from other tests.
"""
import ctypes

import numpy as np
import pytest

import __graft_entry__
from csr_spmm_02_gb300 import gen, spmm
from tests import gpu_helpers as H

SCRATCH_BYTES = 32 << 20  # the library's fixed array
ITEMS_PER_RANGE = 2048    # merge-path items (row ends + nonzeros) per range


def scratch_bytes(M, nnz, N):
    """Bytes of the fixed array a problem needs: error word, range coordinates, carry rows."""
    P = -(-(M + nnz) // ITEMS_PER_RANGE)
    part = -(-8 * (P + 1) // 256) * 256
    return 256 + part + 8 * N * P


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


def test_noalloc_size_limit_is_exact(lib):
    """One range more than the largest problem that fits is refused (before any CUDA call)."""
    N = 2048
    P = max(p for p in range(1, 4096) if scratch_bytes(0, p * ITEMS_PER_RANGE, N) <= SCRATCH_BYTES)
    assert scratch_bytes(0, (P + 1) * ITEMS_PER_RANGE, N) > SCRATCH_BYTES
    M = 64
    big = ctypes.c_void_p(256)
    over = (P + 1) * ITEMS_PER_RANGE - M  # M + nnz fills P + 1 ranges
    assert lib.spmm_csr_f32_noalloc(M, 1024, N, over, big, big, big, big, big, ctypes.c_void_p()) == 3


def _run_noalloc(p, a, C=None, offset_b=0):
    import torch
    B = a["B"]
    if offset_b:  # B starting one float past a 16-byte boundary
        raw = torch.empty(B.numel() + offset_b, dtype=torch.float32, device="cuda")
        B = raw[offset_b:].view(p.K, p.N)
        B.copy_(a["B"])
    if C is None:
        C = torch.full((p.M, p.N), float("nan"), device="cuda")
    spmm.spmm_csr_f32_noalloc(p.M, p.K, p.N, p.nnz, a["rowptr"], a["colind"], a["vals"], B, C)
    assert spmm.spmm_check_device() == 0, "device error word set"
    return C


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_one_call_twice(lib):
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
        C_new = _run_noalloc(p, a)
        C_orc, S = H.reference(p)
        H.assert_within(C_new, C_orc, S, "f32", "noalloc vs oracle")
        H.assert_within(C_new, C_ref.cpu().numpy().astype(np.float64), S, "f32", "noalloc vs one-call")


@pytest.mark.gpu
@pytest.mark.parametrize("N,offset_b", [(3, 0), (13, 0), (64, 1)])
def test_noalloc_scalar_and_misaligned(lib, N, offset_b):
    """N % 4 != 0 and a B that is not 16-byte aligned both take the scalar path."""
    rng = np.random.default_rng(40 + N)
    p = gen.random_csr(rng, 2500, 1200, N, mean_row=9, empty_frac=0.3, long_rows=[(7, 1200)])
    a = H.device_arrays(p)
    for _ in range(2):
        C = _run_noalloc(p, a, offset_b=offset_b)
        C_orc, S = H.reference(p)
        H.assert_within(C, C_orc, S, "f32", f"noalloc N={N} offset={offset_b}")


@pytest.mark.gpu
def test_noalloc_long_row_and_growing_ranges(lib):
    """A 100,000-nonzero row split over many ranges, then a call with more
    ranges than the first on the same stream: no carry row of the earlier call
    may leak into the later one."""
    rng = np.random.default_rng(52)
    small = gen.random_csr(rng, 500, 300, 32, mean_row=5, empty_frac=0.3, long_rows=[(3, 300)])
    big = gen.random_csr(rng, 4000, 120_000, 32, mean_row=10, empty_frac=0.4,
                         long_rows=[(1234, 100_000), (3999, 5000)])
    assert -(-(big.M + big.nnz) // ITEMS_PER_RANGE) > 2 * -(-(small.M + small.nnz) // ITEMS_PER_RANGE)
    for p in (small, big, small, big):
        C = _run_noalloc(p, H.device_arrays(p))
        C_orc, S = H.reference(p)
        H.assert_within(C, C_orc, S, "f32", f"noalloc M={p.M}")


@pytest.mark.gpu
def test_noalloc_scratch_just_fits(lib):
    """The largest problem (in ranges) whose scratch fits the fixed array at N = 2048."""
    import torch
    N, M, K = 2048, 64, 1024
    P = max(p for p in range(1, 4096) if scratch_bytes(0, p * ITEMS_PER_RANGE, N) <= SCRATCH_BYTES)
    nnz = P * ITEMS_PER_RANGE - M
    assert scratch_bytes(M, nnz, N) <= SCRATCH_BYTES < scratch_bytes(M, nnz + ITEMS_PER_RANGE, N)
    rng = np.random.default_rng(77)
    lens = np.full(M, nnz // M, dtype=np.int64)
    lens[: nnz - int(lens.sum())] += 1
    rowptr = gen.rowptr_from_counts(lens)
    colind = rng.integers(0, K, size=nnz).astype(np.int32)  # duplicates are summed
    vals = rng.uniform(-1, 1, nnz).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    p = gen.CsrProblem("just-fits", M, K, N, rowptr, colind, vals, B, "f32")
    C = _run_noalloc(p, H.device_arrays(p))
    H.assert_within_all(C.cpu().numpy(), p, "noalloc just-fits")
    del C
    torch.cuda.empty_cache()


@pytest.mark.gpu
def test_noalloc_nnz_mismatch_is_reported(lib):
    """nnz other than rowptr[M]: no range reads a nonzero, C stays unwritten and
    spmm_check_device returns SPMM_ERR_INVALID_CSR once (then the word is clear)."""
    import torch
    rng = np.random.default_rng(9)
    p = gen.random_csr(rng, 800, 400, 32, mean_row=6, empty_frac=0.2)
    a = H.device_arrays(p)
    for delta in (5, -5):
        pad = torch.zeros(p.nnz + max(delta, 0), dtype=torch.int32, device="cuda")
        pad[: p.nnz] = a["colind"]
        padv = torch.zeros(p.nnz + max(delta, 0), dtype=torch.float32, device="cuda")
        padv[: p.nnz] = a["vals"]
        C = torch.full((p.M, p.N), 7.0, device="cuda")
        spmm.spmm_csr_f32_noalloc(p.M, p.K, p.N, p.nnz + delta, a["rowptr"], pad, padv, a["B"], C)
        assert spmm.spmm_check_device() == 2  # SPMM_ERR_INVALID_CSR
        assert spmm.spmm_check_device() == 0  # read and cleared
        assert bool((C == 7.0).all()), "a rejected call must not write C"
    C = _run_noalloc(p, a)  # the next well-formed call is unaffected
    C_orc, S = H.reference(p)
    H.assert_within(C, C_orc, S, "f32", "noalloc after a rejected call")
