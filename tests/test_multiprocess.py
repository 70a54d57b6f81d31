"""The replicas path of bench.py across ranks, with two gloo ranks on the CPU.

Each rank builds the same level independently (the path shards only by
replication here); the job's time is the slowest rank's and its throughput the
units of all ranks over that time. This checks the cross-rank aggregation the
bench uses, and that the reference arm leaves every rank but 0 without work.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r timed (10 + r) ms in total and reached an end-to-end rate of 100 * (r + 1) per rank
    total, e2e = bench.aggregate_ranks(10.0 + rank, 100.0 * (rank + 1) * world, world, dist, torch.device("cpu"))
    value = bench.job_throughput(world, 5, 1000, total)
    out.put((rank, total, e2e, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, e2e, value in res:
        assert total == 11.0                 # max over ranks
        assert e2e == 100.0 * world          # slowest rank's rate x world
        assert value == pytest.approx(world * 5 * 1000 / 0.011)


def test_reference_arm_other_ranks_do_nothing(capsys):
    import argparse

    import bench
    args = argparse.Namespace(workload="root", steps=1, warmup=3, ref_budget=0.01)
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""
