"""The five benchmark workloads at full size, in the launch configuration the
benchmark times (automatic kernel choice, default range size), plus the other
kernel families.  Every one of the M x N output elements of every kernel is
compared with the CPU oracle (run over row blocks on the host's cores);
whole-matrix properties: finite everywhere, empty rows exactly zero."""
import gc

import numpy as np
import pytest
import torch

from csr_spmm_02_gb300 import gen
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", gen.WORKLOAD_ORDER)
def test_workload_parity(name):
    p = gen.make_workload(name)
    a = H.device_arrays(p)
    expect_kernel = {"uniform1k": "row", "uniform64k": "row", "banded": "window_tc"}.get(name, "balanced")
    others = {"row": ("balanced",), "window_tc": ("window", "row", "balanced"), "balanced": ("row",)}[expect_kernel]
    empty = torch.from_numpy(np.flatnonzero(np.diff(p.rowptr) == 0)).cuda()
    outputs = {}
    for kernel in ("auto",) + others:
        C, plan = H.run(p, kernel=kernel, arrays=a)
        if kernel == "auto":
            assert plan.info()["kernel"] == expect_kernel
        assert bool(torch.isfinite(C).all())
        if len(empty):
            assert not bool(C[empty].any()), "empty rows must be exactly zero"
        outputs[kernel] = C.cpu().numpy()
        plan.destroy()
        del C
    del a
    gc.collect()
    torch.cuda.empty_cache()
    for r0, r1, C_ref, S in H.reference_blocks(p):
        for kernel, C in outputs.items():
            H.assert_within(C[r0:r1], C_ref, S, p.b_dtype, f"{name}/{kernel} rows {r0}..{r1 - 1}")
