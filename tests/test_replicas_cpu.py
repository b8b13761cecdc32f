"""The N > 1 path of bench.py on the CPU: every rank runs an independent
replica and the job's time is the slowest rank's (an all-reduce MAX over a
gloo group of two processes), its throughput every rank's tokens over that
time.  No GPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks([1.5, 2.25][rank], world, torch.device("cpu"))
    out[rank] = (ms, bench.job_tokens_per_s(world, 16384, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms, v = out[r]
        assert ms == 2.25
        assert abs(v - 2 * 16384 / 2.25e-3) < 1e-6 * v


def test_single_rank_needs_no_group():
    import bench
    assert bench.max_over_ranks(3.0, 1, torch.device("cpu")) == 3.0
    assert bench.job_tokens_per_s(1, 1000, 2.0) == 1000 / 2e-3
