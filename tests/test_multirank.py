"""The benchmark's multi-rank path on CPU (gloo, world size 2, 127.0.0.1).

Each rank of `bench.py --gpus N` runs its own replica of the decode-layer
workload (the layer needs no second GPU); the job's throughput is every
rank's streamed bytes over the slowest rank's device time. These tests run
that aggregation and the reference arm's rank rule with two CPU processes.
"""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r streamed (r + 1) GB per step for 10 steps in (r + 1) * 100 ms
        gbs, ms = bench.aggregate_throughput((rank + 1) * 1e9, 10, (rank + 1) * 100.0)
        q.put((rank, gbs, ms, bench.reduce_over_ranks(rank + 0.5, "sum")))
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, gbs, ms, s in out:
        assert ms == 200.0                       # slowest rank
        assert abs(gbs - (1 + 2) * 10 / 0.2) < 1e-9  # 30 GB over 0.2 s
        assert s == 2.0


def test_single_process_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    gbs, ms = bench.aggregate_throughput(1e9, 4, 50.0)
    assert ms == 50.0 and abs(gbs - 80.0) < 1e-12


def test_reference_arm_non_zero_rank_exits_quietly(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup, gpus, seed = 1, 1, 2, 1
    bench.run_reference(A(), rank=1, world=2)
    assert capsys.readouterr().out == ""
