"""The multi-GPU form of the path is replicas only (tokens shard with no exchange), so the N>1
logic is the bench's: every rank times its own replica, the step time is the slowest rank's, and
the job's throughput is the units all ranks processed over that time.  Checked here with two
gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [0.010, 0.014][rank]                     # rank 1 is the slow one
    sec = bench.max_over_ranks(local, dist, torch.device("cpu"))
    value = bench.job_throughput(1000.0, world, sec)
    q.put((rank, sec, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, sec, value in res:
        assert sec == pytest.approx(0.014)
        assert value == pytest.approx(2 * 1000.0 / 0.014)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(0.5, None, None) == 0.5
    assert bench.job_throughput(10.0, 1, 2.0) == 5.0
