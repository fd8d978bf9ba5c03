"""Multi-rank host logic of bench.py on CPU: two gloo ranks (world size 2).

The layer shards over tokens with replicated weights and no exchange (each token's output
depends only on its own row), so the multi-GPU run is N independent replicas; what needs
checking is the host side: rendezvous, barrier, max-over-ranks timing, distinct token shards.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    import workloads as wl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, l = bench.dist_env()
    assert (w, r, l) == (world, rank, rank)
    bench.barrier(world)
    t = bench.max_over_ranks(1.5 + rank, world)          # rank times 1.5 and 2.5 -> 2.5
    shape = wl.WORKLOADS["tiny_f32"]
    x = wl.gen_x(shape, 0 if rank == 0 else 1000 + rank)  # bench's per-rank token shard
    out[rank] = (t, float(x[0, 0]))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert out[0][0] == out[1][0] == 2.5
    assert out[0][1] != out[1][1]          # different tokens on different ranks


def test_weak_scaling_value():
    # value = tokens of all ranks / max-over-ranks device time
    T, steps, world, t_max = 4096, 20, 2, 0.05
    assert T * steps * world / t_max == pytest.approx(3276800.0)
