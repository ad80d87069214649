"""SpMM at the largest nnz the library accepts (SPMM_MAX_EXTENT = 2^31 - 65536).

With M = 2^24 rows the merged sequence of nonzeros and row ends (M + nnz
items) passes 2^31, so the plan's range coordinates, the staging of the last
ranges and the fixup of rows split over hundreds of CTAs all run at the top of
their index range.  Rows are checked against the fp64 oracle on a sample that
holds the first and last rows, every long row, random rows and the rows where
sampled ranges start (the oracle computes rows one by one; the whole matrix
would take it minutes).  The one-call form must give the same C bit for bit,
and one nonzero past the limit must be refused before any kernel reads it.
"""
import numpy as np
import pytest
import torch

import oracle
from csr_spmm_02_gb300 import spmm

MAX_EXTENT = (1 << 31) - 65536


def _rows_of_diagonals(rowptr64, diags):
    """Row holding each merge-path diagonal d: the first row whose end item e(r) = rowptr[r+1] + r is >= d."""
    M = len(rowptr64) - 1
    ends = rowptr64[1:] + np.arange(M, dtype=np.int64)
    return np.minimum(np.searchsorted(ends, diags, side="left"), M - 1)


@pytest.mark.gpu
def test_spmm_at_the_largest_nnz():
    dev = torch.device("cuda")
    free, _ = torch.cuda.mem_get_info()
    if free < (24 << 30):
        pytest.skip("needs 24 GiB of free device memory")
    M, K, N = 1 << 24, 1 << 20, 4
    rng = np.random.default_rng(2031)
    lens = rng.integers(0, 256, M, dtype=np.int64)  # mean 127.5: about 2.139e9 nonzeros, a few empty rows
    long_rows = rng.choice(M, 16, replace=False)
    extra = MAX_EXTENT - int(lens.sum())
    assert extra > 0
    lens[long_rows] += extra // 16
    lens[long_rows[0]] += extra - 16 * (extra // 16)
    rowptr64 = np.zeros(M + 1, np.int64)
    np.cumsum(lens, out=rowptr64[1:])
    assert rowptr64[-1] == MAX_EXTENT and M + MAX_EXTENT > (1 << 31)
    nnz = MAX_EXTENT

    gen = torch.Generator(device=dev)
    gen.manual_seed(2031)
    rowptr = torch.from_numpy(rowptr64.astype(np.int32)).to(dev)
    colind = torch.randint(0, K, (nnz,), dtype=torch.int32, device=dev, generator=gen)
    vals = torch.empty(nnz, dtype=torch.float32, device=dev).uniform_(-1.0, 1.0, generator=gen)
    Bh = rng.standard_normal((K, N)).astype(np.float32)
    B = torch.from_numpy(Bh).to(dev)
    C = torch.full((M, N), float("nan"), device=dev)

    plan = spmm.spmm_csr_plan(rowptr, M, nnz, N)
    info = plan.info()
    assert info["kernel"] == "balanced"
    assert info["nnz"] == nnz and info["max_row_nnz"] == int(lens.max())
    assert info["empty_rows"] == int((lens == 0).sum())
    spmm.spmm_csr_f32_exec(plan, K, colind, vals, B, C)
    torch.cuda.synchronize()
    assert spmm.spmm_plan_check_device(plan) == 0
    T, P = info["items_per_cta"], info["num_ctas"]
    assert P == (M + nnz + T - 1) // T
    plan.destroy()

    # the sample: first and last rows, the long rows, random rows, the rows where
    # sampled ranges start (the last ranges among them)
    cs = np.concatenate([rng.integers(0, P, 600), np.arange(P - 8, P)])
    rows = np.unique(np.concatenate([
        [0, 1, M - 2, M - 1], long_rows, rng.integers(0, M, 2000),
        _rows_of_diagonals(rowptr64, cs.astype(np.int64) * T)]))
    starts, ends = rowptr64[rows], rowptr64[rows + 1]
    idx = np.concatenate([np.arange(s, e, dtype=np.int64) for s, e in zip(starts, ends)])
    idx_d = torch.from_numpy(idx).to(dev)
    sub_col = colind.index_select(0, idx_d).cpu().numpy()
    sub_val = vals.index_select(0, idx_d).cpu().numpy()
    sub_rp = np.concatenate([[0], np.cumsum(ends - starts)]).astype(np.int32)
    ref, S = oracle.spmm_reference(sub_rp, sub_col, sub_val, Bh)
    got = C.index_select(0, torch.from_numpy(rows).to(dev)).double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert (err <= 1e-5 * S + 1e-30).all(), float((err / (S + 1e-30)).max())

    # the one-call form plans the same ranges: the same C, bit for bit
    C2 = torch.full((M, N), float("nan"), device=dev)
    spmm.spmm_csr_f32(M, K, N, rowptr, colind, vals, B, C2)
    torch.cuda.synchronize()
    assert spmm.spmm_check_device() == 0
    assert torch.equal(C, C2)
    del C2

    # one nonzero past the limit: refused by the plan (host check) and by the
    # one-call form once it has read rowptr[M] (before any kernel reads colind)
    with pytest.raises(spmm.SpmmError) as e:
        spmm.spmm_csr_plan(rowptr, M, nnz + 1, N)
    assert e.value.status == 3  # SPMM_ERR_UNSUPPORTED
    rowptr[M] = nnz + 1
    with pytest.raises(spmm.SpmmError) as e:
        spmm.spmm_csr_f32(M, K, N, rowptr, colind, vals, B, C)
    assert e.value.status == 3  # SPMM_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    del colind, vals, C, B, rowptr, idx_d
    torch.cuda.empty_cache()


def _rows_of_diagonals_on_device(rowptr, M, diags):
    """The same search as _rows_of_diagonals, run on the device (rowptr stays there)."""
    lo = torch.zeros_like(diags)
    hi = torch.full_like(diags, M - 1)
    for _ in range(32):
        mid = (lo + hi) // 2
        left = rowptr.index_select(0, mid + 1).long() + mid >= diags
        hi = torch.where(left, mid, hi)
        lo = torch.where(left, lo, torch.minimum(mid + 1, hi))  # stays at M - 1 past the last row end
    return lo


@pytest.mark.gpu
def test_spmm_at_the_largest_m():
    """M = SPMM_MAX_EXTENT rows (2^27 nonzeros scattered over them, most rows
    empty), N = 4: the planner's own kernel and the balanced kernel, each
    checked against the oracle on the first and last rows, random rows, rows
    that hold nonzeros and the rows where sampled ranges start."""
    dev = torch.device("cuda")
    free, _ = torch.cuda.mem_get_info()
    if free < (96 << 30):
        pytest.skip("needs 96 GiB of free device memory")
    M, K, N, nnz = MAX_EXTENT, 1 << 20, 4, 1 << 27
    gen = torch.Generator(device=dev)
    gen.manual_seed(2032)
    # rowptr[r] = number of nonzeros in rows < r, built from the sorted row of
    # every nonzero in chunks (every torch op here stays below 2^31 elements)
    row_of = torch.randint(0, M, (nnz,), device=dev, generator=gen)
    nonempty = row_of[:1000].cpu().numpy()
    row_of = torch.sort(row_of).values
    rowptr = torch.empty(M + 1, dtype=torch.int32, device=dev)
    chunk = 1 << 27
    for r0 in range(0, M + 1, chunk):
        r1 = min(r0 + chunk, M + 1)
        q = torch.arange(r0, r1, dtype=torch.int64, device=dev)
        rowptr[r0:r1] = torch.searchsorted(row_of, q, side="left").to(torch.int32)
    del row_of, q
    torch.cuda.empty_cache()
    assert int(rowptr[0]) == 0 and int(rowptr[M]) == nnz
    colind = torch.randint(0, K, (nnz,), dtype=torch.int32, device=dev, generator=gen)
    vals = torch.empty(nnz, dtype=torch.float32, device=dev).uniform_(-1.0, 1.0, generator=gen)
    rng = np.random.default_rng(2032)
    Bh = rng.standard_normal((K, N)).astype(np.float32)
    B = torch.from_numpy(Bh).to(dev)
    C = torch.empty((M, N), dtype=torch.float32, device=dev)

    for kernel in ("auto", "balanced"):
        C.fill_(float("nan"))
        plan = spmm.spmm_csr_plan(rowptr, M, nnz, N, kernel=kernel)
        info = plan.info()
        assert info["nnz"] == nnz and info["M"] == M
        spmm.spmm_csr_f32_exec(plan, K, colind, vals, B, C)
        torch.cuda.synchronize()
        assert spmm.spmm_plan_check_device(plan) == 0
        parts = [np.array([0, 1, M - 2, M - 1]), rng.integers(0, M, 3000), nonempty]
        if info["kernel"] == "balanced":
            T, P = info["items_per_cta"], info["num_ctas"]
            assert P == (M + nnz + T - 1) // T
            cs = np.concatenate([rng.integers(0, P, 600), np.arange(P - 8, P)]).astype(np.int64)
            parts.append(_rows_of_diagonals_on_device(rowptr, M, torch.from_numpy(cs * T).to(dev)).cpu().numpy())
        plan.destroy()
        rows = np.unique(np.concatenate(parts)).astype(np.int64)
        rows_d = torch.from_numpy(rows).to(dev)
        starts = rowptr.index_select(0, rows_d).long().cpu().numpy()
        ends = rowptr.index_select(0, rows_d + 1).long().cpu().numpy()
        idx = np.concatenate([np.arange(s, e, dtype=np.int64) for s, e in zip(starts, ends)])
        idx_d = torch.from_numpy(idx).to(dev)
        sub_col = colind.index_select(0, idx_d).cpu().numpy()
        sub_val = vals.index_select(0, idx_d).cpu().numpy()
        sub_rp = np.concatenate([[0], np.cumsum(ends - starts)]).astype(np.int32)
        ref, S = oracle.spmm_reference(sub_rp, sub_col, sub_val, Bh)
        got = torch.stack([C[int(r)] for r in rows]).double().cpu().numpy()  # views: no index kernel over all of C
        assert np.isfinite(got).all(), info["kernel"]
        err = np.abs(got - ref)
        assert (err <= 1e-5 * S + 1e-30).all(), (info["kernel"], float((err / (S + 1e-30)).max()))
    del colind, vals, C, B, rowptr
    torch.cuda.empty_cache()
