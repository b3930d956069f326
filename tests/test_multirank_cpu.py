"""The benchmark's multi-GPU path on CPU: two gloo ranks, each an independent
replica, aggregated as slowest-rank time and summed units (no data exchange:
the layer's replicas share nothing)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        local_s = 1.0 + rank  # rank 1 is the slower replica
        units = 100.0 * (rank + 1)
        bench.barrier(world)
        max_s, total = bench.aggregate(local_s, units, world, device=None)
        q.put((rank, max_s, total))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, max_s, total in got:
        assert max_s == pytest.approx(2.0)
        assert total == pytest.approx(300.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import json

    import bench

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1"]) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["workload"] == "skinny_m16_k4096_n4096_bf16"
