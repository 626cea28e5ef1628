"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the timed
region's max over ranks and the whole-job byte count, plus the replicas'
independent seeds."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    secs, nbytes = bench.aggregate(1.0 + rank, 1000 * (rank + 1))
    env = bench.dist_env()
    dist.destroy_process_group()
    q.put((rank, secs, nbytes, env))


def test_aggregate_two_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, secs, nbytes, env in res:
        assert secs == 2.0  # slowest rank
        assert nbytes == 3000  # all ranks' work
        assert env == (world, rank, rank)


def test_single_process_aggregate_is_identity():
    import bench

    assert bench.aggregate(1.5, 77) == (1.5, 77)


def test_reference_arm_other_ranks_exit_quietly(capsys, monkeypatch):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        warmup_ref = 0
        steps_ref = 1

    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""
