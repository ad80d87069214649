"""CUDA path vs the CPU oracle on small seeded inputs (several tiles, split
rows, ragged tails, edge cases).  Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

from csr_spmm_02_gb300 import gen, spmm
from tests import gpu_helpers as H
from tests import oracle_pins

pytestmark = pytest.mark.gpu

KERNELS = ["row", "balanced", "window", "smalln"]


def mixed(seed, M=1500, K=900, N=64, b_dtype="f32", integer=False, duplicates=False):
    rng = np.random.default_rng(seed)
    return gen.random_csr(rng, M, K, N, mean_row=10, empty_frac=0.3, long_rows=[(7, K), (M - 3, 600)],
                          b_dtype=b_dtype, integer=integer, duplicates=duplicates)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("b_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 3, 4, 8, 12, 32, 33, 64, 100, 128, 256, 520])
def test_random_parity(kernel, b_dtype, N):
    p = mixed(N, N=N, b_dtype=b_dtype)
    C, _ = H.run(p, kernel=kernel, items_per_cta=256)
    C_ref, S = H.reference(p)
    H.assert_within(C, C_ref, S, b_dtype, f"{kernel}/{b_dtype}/N={N}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("b_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [8, 64, 256])
def test_integer_inputs_exact(kernel, b_dtype, N):
    """Small integers: every partial sum is exact in fp32, so any order gives the exact result."""
    p = mixed(100 + N, N=N, b_dtype=b_dtype, integer=True, duplicates=True)
    C, _ = H.run(p, kernel=kernel, items_per_cta=256)
    C_ref, _ = H.reference(p)
    H.assert_exact(C, C_ref, f"{kernel}/{b_dtype}/N={N}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_special_matrices_exact(kernel):
    rng = np.random.default_rng(3)
    n, N = 1000, 64
    B = gen.uniform_b(rng, n, N)
    for (rp, ci, v), expect in (
        (gen.identity_csr(n), B),
        (gen.identity_csr(n, 2.0 ** -5), B * 2.0 ** -5),
        (gen.permutation_csr(perm := rng.permutation(n)), B[perm]),
    ):
        p = gen.CsrProblem("special", n, n, N, rp, ci, v, B, "f32")
        C, _ = H.run(p, kernel=kernel, items_per_cta=256)
        H.assert_exact(C, expect.astype(np.float64), kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("b_dtype", ["f32", "bf16"])
def test_hand_worked_4x4(kernel, b_dtype):
    g = oracle_pins.load_golden_hand_4x4()
    B = g["B"].astype(np.float32)
    if b_dtype == "bf16":
        B = gen.f32_to_bf16_bits(B)  # small integers are exact in bf16
    p = gen.CsrProblem("hand", 4, 4, 2, g["rowptr"].astype(np.int32), g["colind"].astype(np.int32),
                       g["vals"].astype(np.float32), B, b_dtype)
    C, _ = H.run(p, kernel=kernel, items_per_cta=256)
    H.assert_exact(C, g["C"], f"{kernel}/{b_dtype}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_edge_cases(kernel):
    rng = np.random.default_rng(8)
    cases = []
    # M = 1 with a few nonzeros; M = 1 empty
    cases.append(gen.CsrProblem("m1", 1, 10, 16, np.array([0, 5], np.int32), np.array([0, 2, 4, 6, 9], np.int32),
                                rng.uniform(-1, 1, 5).astype(np.float32), gen.uniform_b(rng, 10, 16), "f32"))
    cases.append(gen.CsrProblem("m1e", 1, 10, 16, np.array([0, 0], np.int32), np.zeros(0, np.int32),
                                np.zeros(0, np.float32), gen.uniform_b(rng, 10, 16), "f32"))
    # nnz = 0 over many rows: C must be overwritten with zeros
    cases.append(gen.CsrProblem("nnz0", 3000, 50, 33, np.zeros(3001, np.int32), np.zeros(0, np.int32),
                                np.zeros(0, np.float32), gen.uniform_b(rng, 50, 33), "f32"))
    # one row holds every nonzero (longer than many CTA ranges), the rest empty
    L = 100000
    rp = np.zeros(401, np.int32)
    rp[201:] = L
    cases.append(gen.CsrProblem("onelong", 400, 120000, 32, rp,
                                np.sort(rng.choice(120000, L, replace=False)).astype(np.int32),
                                rng.uniform(-1, 1, L).astype(np.float32), gen.uniform_b(rng, 120000, 32), "f32"))
    # K = 1, every row uses column 0
    cases.append(gen.CsrProblem("k1", 500, 1, 8, np.arange(501, dtype=np.int32), np.zeros(500, np.int32),
                                rng.uniform(-1, 1, 500).astype(np.float32), gen.uniform_b(rng, 1, 8), "f32"))
    for p in cases:
        C, _ = H.run(p, kernel=kernel, items_per_cta=256)
        C_ref, S = H.reference(p)
        H.assert_within(C, C_ref, S, "f32", f"{kernel}/{p.name}")


def test_zero_sized_is_noop():
    for M, N in ((0, 8), (5, 0)):
        rowptr = torch.zeros(M + 1, dtype=torch.int32, device="cuda")
        C = torch.full((M, N), 7.0, device="cuda")
        plan = spmm.spmm_csr_plan(rowptr, M, 0, N)
        spmm.spmm_csr_f32_exec(plan, 4, None, None, None, C)
        torch.cuda.synchronize()
        assert bool((C == 7.0).all())


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("b_dtype", ["f32", "bf16"])
def test_misaligned_pointers(kernel, b_dtype):
    """B, C, colind and vals at offsets that break 16-byte alignment: scalar B
    path and plain (non-bulk) staging, same results."""
    p = mixed(77, N=64, b_dtype=b_dtype)
    a = H.device_arrays(p)
    def shifted(t):
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
        v = buf[1:].view(t.shape)
        v.copy_(t)
        return v
    a = {k: shifted(v) if k != "rowptr" else v for k, v in a.items()}
    Cbuf = torch.full((p.M * p.N + 1,), float("nan"), device="cuda")
    C = Cbuf[1:].view(p.M, p.N)
    C, _ = H.run(p, kernel=kernel, items_per_cta=256, arrays=a, C=C)
    C_ref, S = H.reference(p)
    H.assert_within(C, C_ref, S, b_dtype, f"misaligned {kernel}/{b_dtype}")


@pytest.mark.parametrize("T", [256, 512, 2048, 8192])
def test_items_per_cta(T):
    p = mixed(55, N=32)
    C, plan = H.run(p, kernel="balanced", items_per_cta=T)
    info = plan.info()
    assert info["items_per_cta"] == T and info["num_ctas"] == -(-(p.M + p.nnz) // T)
    C_ref, S = H.reference(p)
    H.assert_within(C, C_ref, S, "f32", f"T={T}")
    q = mixed(56, N=32, integer=True)
    C, _ = H.run(q, kernel="balanced", items_per_cta=T)
    H.assert_exact(C, H.reference(q)[0], f"integer T={T}")


@pytest.mark.parametrize("N", [1, 2, 3, 4, 8, 12, 24, 32, 64])
def test_default_items_per_cta(N):
    """The plan's own range size: 3072 items for 8 < N <= 32, 3840 for N = 1, 3, 4, 8, else 2048."""
    p = mixed(57, M=6000, K=3000, N=N)
    C, plan = H.run(p, kernel="balanced")
    info = plan.info()
    T = 3072 if 8 < N <= 32 else 3840 if N in (1, 3, 4, 8) else 2048
    assert info["items_per_cta"] == T and info["num_ctas"] == -(-(p.M + p.nnz) // T)
    C_ref, S = H.reference(p)
    H.assert_within(C, C_ref, S, "f32", f"default T, N={N}")
    q = mixed(58, M=6000, K=3000, N=N, integer=True)
    C, _ = H.run(q, kernel="balanced")
    H.assert_exact(C, H.reference(q)[0], f"integer, default T, N={N}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_deterministic(kernel):
    p = mixed(91, N=128)
    C1, plan = H.run(p, kernel=kernel, items_per_cta=512)
    a = H.device_arrays(p)
    C2, _ = H.run(p, arrays=a, plan=plan)
    assert torch.equal(C1, C2)


def test_validate():
    p = mixed(5, N=4)
    a = H.device_arrays(p)
    assert spmm.spmm_csr_validate(a["rowptr"], a["colind"], p.M, p.K, p.nnz) == 0
    bad = a["colind"].clone()
    bad[17] = p.K
    assert spmm.spmm_csr_validate(a["rowptr"], bad, p.M, p.K, p.nnz) == 2
    bad = a["rowptr"].clone()
    bad[10] = bad[11] + 1
    assert spmm.spmm_csr_validate(bad, a["colind"], p.M, p.K, p.nnz) == 2
    assert spmm.spmm_csr_validate(a["rowptr"], a["colind"], p.M, p.K, p.nnz + 1) == 2


@pytest.mark.parametrize("b_dtype", ["f32", "bf16"])
def test_one_call_form_matches_plan_exec(b_dtype):
    for seed, uniform in ((1, True), (2, False)):
        rng = np.random.default_rng(seed)
        if uniform:
            rp, ci = gen.uniform_structure(rng, 2000, 1500, 20)
            p = gen.CsrProblem("u", 2000, 1500, 64, rp, ci, rng.uniform(-1, 1, len(ci)).astype(np.float32),
                               gen.uniform_b(rng, 1500, 64, b_dtype), b_dtype)
        else:
            p = mixed(seed, N=64, b_dtype=b_dtype)
        a = H.device_arrays(p)
        C_plan, plan = H.run(p, arrays=a)
        C_one = torch.full_like(C_plan, float("nan"))
        f = spmm.spmm_csr_f32 if b_dtype == "f32" else spmm.spmm_csr_bf16f32
        f(p.M, p.K, p.N, a["rowptr"], a["colind"], a["vals"], a["B"], C_one)
        torch.cuda.synchronize()
        assert torch.equal(C_plan, C_one)
        assert plan.info()["kernel"] == ("row" if uniform else "balanced")


def test_one_call_pool_reuse_and_release():
    """Repeated one-call products reuse the pool's blocks; after a release the next call maps new
    memory and gives the same bits.  A negative rowptr[M] is rejected as an invalid CSR."""
    p = mixed(5, N=64)
    a = H.device_arrays(p)
    C_ref, S = H.reference(p)
    outs = []
    for i in range(4):
        C = torch.full((p.M, p.N), float("nan"), device="cuda")
        spmm.spmm_csr_f32(p.M, p.K, p.N, a["rowptr"], a["colind"], a["vals"], a["B"], C)
        if i == 1:
            torch.cuda.synchronize()
            spmm.spmm_pool_release()
        outs.append(C)
    torch.cuda.synchronize()
    H.assert_within(outs[0], C_ref, S, "f32", "one-call")
    for C in outs[1:]:
        assert torch.equal(C, outs[0])
    bad = a["rowptr"].clone()
    bad[-1] = -5
    C = torch.empty((p.M, p.N), device="cuda")
    with pytest.raises(spmm.SpmmError) as err:
        spmm.spmm_csr_f32(p.M, p.K, p.N, bad, a["colind"], a["vals"], a["B"], C)
    assert err.value.status == 2  # SPMM_ERR_INVALID_CSR


def test_side_stream():
    p = mixed(12, N=32)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = H.device_arrays(p)
        C = torch.empty((p.M, p.N), device="cuda")
        C, _ = H.run(p, kernel="balanced", arrays=a, C=C, stream=s)
    C_ref, S = H.reference(p)
    H.assert_within(C, C_ref, S, "f32", "side stream")


@pytest.mark.parametrize("kernel", ["row", "balanced"])
@pytest.mark.parametrize("b_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cap", [8, 32, 64])
def test_column_tile_cap(kernel, b_dtype, cap):
    """N-slicing: the same results with the column tile capped (several tiles in grid.y)."""
    p = mixed(7 + cap, N=256, b_dtype=b_dtype)
    a = H.device_arrays(p)
    plan = spmm.spmm_csr_plan(a["rowptr"], p.M, p.nnz, p.N, kernel=kernel, items_per_cta=256)
    spmm.spmm_plan_set_column_tile(plan, cap)
    assert plan.info()["column_tile"] == cap
    C, _ = H.run(p, arrays=a, plan=plan)
    C_ref, S = H.reference(p)
    H.assert_within(C, C_ref, S, b_dtype, f"{kernel}/{b_dtype}/cap={cap}")
    with pytest.raises(spmm.SpmmError):
        spmm.spmm_plan_set_column_tile(plan, -1)

