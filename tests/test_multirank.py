"""bench.py's multi-rank logic on CPU with gloo ranks: the whole-job rate is
all ranks' work over the slowest rank's time; the row-block split of one A
(the library's spmm_csr_row_blocks, rows kept whole, B replicated) covers
every row exactly once and the ranks' oracle outputs, concatenated, equal the
whole problem's oracle output bitwise; the reference arm runs on rank 0
only."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rate, slowest = bench.whole_job_rate(local_work=10.0 * (rank + 1), local_seconds=1.0 + rank)
        out[rank] = (rate, slowest, bench.reduce_max(float(rank)), bench.dist_env())
    finally:
        dist.destroy_process_group()


def test_whole_job_rate_two_gloo_ranks():
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    for rank in (0, 1):
        rate, slowest, mx, env = out[rank]
        assert slowest == 2.0 and rate == pytest.approx(30.0 / 2.0) and mx == 1.0
        assert env == (2, rank, rank)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    import json
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    assert bench.main(["--impl", "reference", "--workload", "uniform1k", "--steps", "2", "--warmup", "1"]) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == "uniform1k" and line["config"]["nnz"] == 16384


def _shard_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import numpy as np
    import bench
    import oracle
    from csr_spmm_02_gb300 import gen
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # every rank builds the same seeded problem (B replicated); skewed rows,
        # one of them longer than a whole rank's share
        p = gen.random_csr(np.random.default_rng(11), 3000, 2500, 12, mean_row=7, empty_frac=0.35,
                           long_rows=[(17, 2500), (2999, 900)])
        sub, r0 = bench.shard_rows(p, rank, world)
        C, _ = oracle.spmm_reference(sub.rowptr, sub.colind, sub.vals, sub.B)
        pieces = [None] * world
        dist.all_gather_object(pieces, (r0, sub.M, sub.nnz, C))
        if rank == 0:
            full, _ = oracle.spmm_reference(p.rowptr, p.colind, p.vals, p.B)
            out["pieces"] = [(a, m, z) for a, m, z, _ in pieces]
            out["equal"] = bool(np.array_equal(np.concatenate([c for *_, c in pieces]), full))
            out["M"], out["nnz"] = p.M, p.nnz
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_row_block_split_gloo(world):
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_shard_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    pieces = out["pieces"]
    starts = [a for a, _, _ in pieces]
    assert starts[0] == 0 and all(a + m == b for (a, m, _), b in zip(pieces, starts[1:] + [out["M"]]))
    assert sum(z for *_, z in pieces) == out["nnz"]  # every nonzero on exactly one rank
    assert out["equal"], "the ranks' row blocks do not reassemble the whole product"


def test_row_blocks_balance_and_edge_cases():
    import numpy as np
    from csr_spmm_02_gb300 import gen, spmm
    rng = np.random.default_rng(4)
    p = gen.random_csr(rng, 20000, 5000, 4, mean_row=9, empty_frac=0.4)
    for parts in (1, 2, 5, 8):
        rs = spmm.spmm_csr_row_blocks(p.rowptr, parts)
        assert rs[0] == 0 and rs[-1] == p.M and np.all(np.diff(rs) >= 0)
        items = np.diff(p.rowptr[rs].astype(np.int64)) + np.diff(rs)  # nonzeros + row ends per block
        share = (p.M + p.nnz) / parts
        # each boundary sits within one row (its nonzeros and its end) of the exact diagonal
        assert items.sum() == p.M + p.nnz
        assert np.all(np.abs(items - share) <= 2 * (np.diff(p.rowptr).max() + 1) + 1)
    # a row longer than a whole share: the block boundary moves to its end, some blocks stay empty
    rp = np.array([0, 1, 1001, 1002, 1003], np.int32)
    rs = spmm.spmm_csr_row_blocks(rp, 4)
    assert rs[0] == 0 and rs[-1] == 4 and np.all(np.diff(rs) >= 0)
    assert spmm.spmm_csr_row_blocks(np.zeros(1, np.int32), 3).tolist() == [0, 0, 0, 0]  # M = 0
    with pytest.raises(spmm.SpmmError):
        spmm.spmm_csr_row_blocks(np.array([0, 5, 3], np.int32), 2)  # decreasing rowptr
    with pytest.raises(spmm.SpmmError):
        spmm.spmm_csr_row_blocks(np.array([1, 5], np.int32), 2)  # rowptr[0] != 0
    with pytest.raises(spmm.SpmmError):
        spmm.spmm_csr_row_blocks(p.rowptr, 0)
