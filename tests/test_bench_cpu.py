"""bench.py's host-side pieces on CPU: the compulsory bytes and flops of each
operation, the reference arm for every operation and option (B redrawn in
bf16 among them), and the per-kernel source hashes that key the traffic
records."""
import json

import numpy as np
import pytest

import bench
from csr_spmm_02_gb300 import gen


def test_op_bytes_and_flops():
    p = gen.make_workload("uniform1k")
    M, K, N, nnz = p.M, p.K, p.N, p.nnz
    assert bench.op_bytes(p, "spmm") == 4 * (M + 1) + 8 * nnz + 4 * K * N + 4 * M * N
    assert bench.op_bytes(p, "sddmm") == 4 * (M + 1) + 4 * nnz + 4 * M * N + 4 * K * N + 4 * nnz
    assert bench.op_bytes(p, "fusedmm") == 4 * (M + 1) + 4 * nnz + 4 * M * N + 8 * K * N + 4 * M * N
    assert bench.op_flops(p, "spmm") == bench.op_flops(p, "sddmm") == 2 * nnz * N
    assert bench.op_flops(p, "fusedmm") == 4 * nnz * N


def test_gather_bytes():
    p = gen.make_workload("uniform1k")  # fp32 B, N = 32
    assert bench.op_gather_bytes(p, "spmm", "row") == p.nnz * p.N * 4
    assert bench.op_gather_bytes(p, "sddmm", "balanced") == p.nnz * p.N * 4
    assert bench.op_gather_bytes(p, "fusedmm", "fusedmm") == 2 * p.nnz * p.N * 4
    assert bench.op_gather_bytes(p, "spmm", "window_tc") is None


def test_dense_operands_are_seeded_fp32():
    p = gen.make_workload("uniform1k")
    C1, B1, D1 = bench.op_dense_inputs(p, "fusedmm")
    C2, B2, D2 = bench.op_dense_inputs(p, "fusedmm")
    assert C1.dtype == np.float32 and C1.shape == (p.M, p.N) and D1.shape == (p.K, p.N)
    assert np.array_equal(C1, C2) and np.array_equal(D1, D2) and np.array_equal(B1, p.B)
    q = gen.random_csr(np.random.default_rng(1), 50, 40, 24, b_dtype="bf16")
    _, Bq, _ = bench.op_dense_inputs(q, "sddmm")  # bf16 B widened exactly
    assert Bq.dtype == np.float32
    assert np.array_equal((q.B.astype(np.uint32) << 16).view(np.float32), Bq)


@pytest.mark.parametrize("argv", [
    ["--op", "sddmm"], ["--op", "fusedmm"], ["--semiring", "min,add"], ["--n", "4"],
    ["--n", "4", "--semiring", "max,mul"], ["--n", "8", "--b-dtype", "bf16"], ["--b-dtype", "bf16"],
])
def test_reference_arm_lines(argv, capsys):
    assert bench.main(["--impl", "reference", "--workload", "uniform1k", "--steps", "1", "--warmup", "0"] + argv) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    if "--n" in argv:
        assert line["config"]["N"] == int(argv[argv.index("--n") + 1])
    if "--b-dtype" in argv:  # B redrawn in bf16: the compulsory bytes count 2-byte B elements
        cfg = line["config"]
        assert cfg["b_dtype"] == "bf16" and "in bf16" in cfg["workload"]
        p = gen.make_workload("uniform1k")
        assert cfg["compulsory_bytes"] == 4 * (p.M + 1) + 8 * p.nnz + 2 * p.K * cfg["N"] + 4 * p.M * cfg["N"]


def test_b_dtype_is_refused_for_sddmm_and_fusedmm():
    for op in ("sddmm", "fusedmm"):
        with pytest.raises(SystemExit):
            bench.main(["--impl", "reference", "--workload", "uniform1k", "--op", op, "--b-dtype", "bf16",
                        "--steps", "1", "--warmup", "0"])


def test_traffic_records_match_their_kernels():
    rec = json.load(open(bench.TRAFFIC_FILE))
    for workload, kernels in rec["captures"].items():
        for kernel, r in kernels.items():
            assert kernel in bench.KERNEL_SOURCES
            if r["source_hash"] == bench.kernel_source_hash(kernel):
                assert bench.ncu_traffic(workload, kernel) == r["dram_bytes_per_launch"]
            else:
                assert bench.ncu_traffic(workload, kernel) is None
