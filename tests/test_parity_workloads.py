"""The five benchmark workloads at full size, in the launch configuration the
benchmark times (automatic kernel choice, default range size), plus the other
kernel family.  Rows are sampled: every row for the two uniform workloads;
otherwise random rows, the longest rows and the rows that CTA range
boundaries cut.  Whole-matrix properties: finite everywhere, empty rows exactly
zero."""
import gc

import numpy as np
import pytest
import torch

from csr_spmm_02_gb300 import gen
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

PLAN_TS = (2048, 3072)  # the plan's default range sizes (N > 32, N <= 32)


def boundary_rows(rowptr, T, limit=3000):
    """Rows containing the start of a merge-path range of T items."""
    M = len(rowptr) - 1
    ends = rowptr[1:].astype(np.int64) + np.arange(M)
    diags = np.arange(0, M + int(rowptr[-1]), T, dtype=np.int64)
    rows = np.searchsorted(ends, diags, side="left")
    rows = np.unique(rows[rows < M])
    return rows[:: max(1, len(rows) // limit)]


def sample_rows(p, rng):
    if p.M <= 70000:
        return None
    lens = np.diff(p.rowptr)
    longest = np.argsort(lens)[-64:]
    rand = rng.choice(p.M, 6000, replace=False)
    return np.unique(np.concatenate([longest, rand, *[boundary_rows(p.rowptr, T) for T in PLAN_TS], [0, p.M - 1]])).astype(np.int32)


@pytest.mark.parametrize("name", gen.WORKLOAD_ORDER)
def test_workload_parity(name):
    p = gen.make_workload(name)
    rng = np.random.default_rng(99)
    rows = sample_rows(p, rng)
    C_ref, S = H.reference(p, rows=rows)
    a = H.device_arrays(p)
    expect_kernel = {"uniform1k": "row", "uniform64k": "row", "banded": "window_tc"}.get(name, "balanced")
    others = {"row": ("balanced",), "window_tc": ("window", "row", "balanced"), "balanced": ("row",)}[expect_kernel]
    for kernel in ("auto",) + others:
        C, plan = H.run(p, kernel=kernel, arrays=a)
        if kernel == "auto":
            assert plan.info()["kernel"] == expect_kernel
        assert bool(torch.isfinite(C).all())
        empty = torch.from_numpy(np.flatnonzero(np.diff(p.rowptr) == 0)).cuda()
        if len(empty):
            assert not bool(C[empty].any()), "empty rows must be exactly zero"
        got = C if rows is None else C[torch.from_numpy(rows.astype(np.int64)).cuda()]
        H.assert_within(got, C_ref, S, p.b_dtype, f"{name}/{kernel}")
        plan.destroy()
        del C
    del a
    gc.collect()
    torch.cuda.empty_cache()
