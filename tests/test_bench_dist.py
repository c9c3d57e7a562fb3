"""The multi-rank bookkeeping of bench.py on CPU: two gloo ranks, each with
its own replica's timing; the job throughput uses the slowest rank's time and
counts every rank's tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t_rank = [0.5, 0.8][rank]  # seconds for 10 steps on this rank
    value, t_all = bench.aggregate(t_rank, world, tokens_per_rank=64, steps=10, dist=dist,
                                   device="cpu")
    out[rank] = (value, t_all)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_uses_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        value, t_all = out[r]
        assert t_all == pytest.approx(0.8)
        assert value == pytest.approx(2 * 64 * 10 / 0.8)


def test_single_rank_aggregation():
    import bench
    value, t_all = bench.aggregate(0.25, 1, 64, 10)
    assert t_all == 0.25 and value == pytest.approx(64 * 10 / 0.25)
