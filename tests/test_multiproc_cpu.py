"""The multi-rank path of bench.py on CPU: two gloo ranks, each with its own replica time;
the reported time is the slowest rank's and the throughput counts every rank's tokens."""
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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = 100.0 + 50.0 * rank            # rank 1 is slower
    t_max = bench.reduce_max(t)
    out[rank] = t_max
    out[world + rank] = bench.throughput(world, 10, 8192, t_max)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    out = mp.get_context("spawn").Array("d", 2 * world)
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0] == out[1] == 150.0
    assert out[2] == out[3] == 2 * 10 * 8192 / 0.150


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max(12.5) == 12.5
    assert bench.throughput(1, 4, 1000, 2000.0) == 2000.0
