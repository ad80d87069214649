"""bench.py's multi-rank logic on CPU: two gloo ranks, each timing an
independent replica; the whole-job rate is all ranks' work over the slowest
rank's time, and the reference arm runs on rank 0 only."""
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
