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


def test_reference_arm_line_carries_the_contract_keys(capsys):
    # Rank 0 of the reference arm (the oracle on the host cores) prints one
    # JSON line with the keys of the GPU arm's line, the same `config`, and
    # a cpu_baseline / e2e describing its own run (a small row sample here).
    import json

    import bench

    class A:
        workload = bench.DEFAULT
        cpu_rows = 16
        warmup = 0
        steps = 1
        cpu_budget_s = 30.0
    bench.run_reference(A(), rank=0, world=1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is False and line["value"] > 0
    assert line["config"] == bench.layer_config(bench.DEFAULT, 1)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
