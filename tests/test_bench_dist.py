"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Ranks run independent replicas (the path shards by sequence; no collective on
the data path): each draws its own seed, the whole-job time is the slowest
rank's, and the job throughput counts every rank's cycles.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [10.0, 12.5][rank]
    out[rank] = (bench.max_over_ranks(ms), bench.rank_seed(42, rank))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    import bench
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == 12.5 and out[1][0] == 12.5
    assert out[0][1] != out[1][1]
    assert bench.job_throughput(world, 100, 12.5) == pytest.approx(2 * 100 / 0.0125)
    assert bench.max_over_ranks(3.0) == 3.0  # no process group: identity
