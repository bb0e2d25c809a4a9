"""The replicas path of bench.py with two ranks on the CPU (gloo): every rank
steps its own layer, the job time is the max over ranks, only rank 0 reports."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        mine = 10.0 * (rank + 1)                      # this rank's timed total
        job = bench.max_over_ranks(mine, world)
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.replica_seed(rank))
        q.put((rank, job, seeds))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_distinct_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, job, seeds in res:
        assert job == 20.0                            # the slowest rank
        assert len(set(seeds)) == 2                   # independent replicas


def test_reference_arm_other_ranks_do_no_work(capsys):
    import bench

    class A:
        workload = bench.DEFAULT
        cpu_rows = 8
        warmup = 0
        steps = 1
        cpu_budget_s = 1.0
    bench.run_reference(A(), rank=1, world=2)
    assert capsys.readouterr().out == ""
