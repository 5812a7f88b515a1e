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


def _replica_layer(O, w):
    """The whole layer on one replica's inputs: router scores, top-k, forward, backward."""
    import numpy as np
    logits = O.router_logits(O.as_f64(w.x), O.as_f64(w.w_r)).astype(np.float32)
    idx, gate = O.route_topk(O.selection_scores(logits, w.bias.numpy()), w.cfg["k"])
    x = O.as_f64(w.x)
    w13, w2, ws13, ws2 = (O.as_f64(t) for t in (w.w13, w.w2, w.ws13, w.ws2))
    fwd = O.layer_forward(x, idx, gate, w13, w2, ws13, ws2)
    g = O.layer_backward(x, idx, gate, fwd, O.as_f64(w.dy), w13, w2, ws13, ws2, w_r=O.as_f64(w.w_r))
    return fwd, g


def _layer_worker(rank, world, port, out):
    """One replica of the layer on CPU: this rank's token batch through the oracle's forward
    and backward, then the ranks compare what they hold over gloo."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np

    import oracle as O
    from synth import make_workload, shrink
    w = make_workload(shrink("pangu_bf16", T=24, d=64, E=8, k=2, f=64, f_s=64), replica=rank)
    fwd, g = _replica_layer(O, w)
    f64 = O.as_f64
    mine = {"x": float(np.abs(f64(w.x)).sum()), "w13": float(np.abs(f64(w.w13)).sum()),
            "y": float(np.abs(fwd["y"]).sum()), "dw13": float(np.abs(g["dw13"]).sum())}
    every = [None] * world
    dist.all_gather_object(every, mine)
    t_max = __import__("bench").reduce_max(10.0 + rank)
    if rank == 0:
        out[0] = float(every[0]["w13"] == every[1]["w13"])          # same weights
        out[1] = float(every[0]["x"] != every[1]["x"])              # own tokens
        out[2] = float(every[0]["y"] != every[1]["y"] and every[0]["dw13"] != every[1]["dw13"])
        out[3] = every[1]["y"]
        out[4] = every[1]["dw13"]
        out[5] = t_max
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_run_the_layer_on_their_own_tokens():
    """Data-parallel replicas: both ranks hold the same weights and their own seeded tokens,
    each runs the whole layer (the fp64 oracle on CPU), and what rank 1 computed in its own
    process equals the same replica computed here; the step time is the slower rank's."""
    import numpy as np

    import oracle as O
    from synth import make_workload, shrink
    world = 2
    out = mp.get_context("spawn").Array("d", 6)
    mp.start_processes(_layer_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0] == 1.0 and out[1] == 1.0 and out[2] == 1.0
    w = make_workload(shrink("pangu_bf16", T=24, d=64, E=8, k=2, f=64, f_s=64), replica=1)
    fwd, g = _replica_layer(O, w)
    assert out[3] == float(np.abs(fwd["y"]).sum())
    assert out[4] == float(np.abs(g["dw13"]).sum())
    assert out[5] == 11.0
