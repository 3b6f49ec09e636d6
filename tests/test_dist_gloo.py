"""The multi-GPU bench path on CPU: world size 2 over gloo.  Each rank plans its own
forest (weak scaling, no data exchange); the bench reduces compact tokens by sum and
step time by max across ranks."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from prefix_shared_chunkwise_gb300.api import Plan
        parent, seg_len, seed = bench.forest_for_rank("fb64k_bf16", rank)
        pl = Plan(parent, seg_len, 64)
        C_all, ms = bench.reduce_across_ranks(pl.info["C"], 10.0 + rank, "cpu")
        out[rank] = (pl.info["C"], seed, C_all, ms, int(parent.sum()))
    finally:
        dist.destroy_process_group()


def test_two_rank_weak_scaling_reduction():
    from prefix_shared_chunkwise_gb300 import build
    build.build()
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    (c0, s0, a0, m0, p0), (c1, s1, a1, m1, p1) = out[0], out[1]
    assert s0 != s1 and (c0 != c1 or p0 != p1)          # distinct forests per rank
    assert a0 == a1 == c0 + c1                           # whole-job tokens
    assert m0 == m1 == 11.0                              # slowest rank's step time
