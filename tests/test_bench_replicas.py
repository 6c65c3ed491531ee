"""Host logic of bench.py's multi-GPU mode, on CPU with two gloo ranks: each replica gets
its own tokens (rank 0 the canonical batch), and the timing reduces to the maximum over
ranks.  (The data path has no collective: replicas are independent.)"""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.5 + rank * 2.25)
        w = bench.replica_workload("decode", rank)
        out[rank] = (t, w.x_seed, w.T)
    finally:
        dist.destroy_process_group()


def test_replicas_and_max_timing_gloo_world2():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 3.75          # max over ranks, on every rank
    assert res[0][1] != res[1][1]                   # different tokens per replica
    assert res[0][2] == res[1][2] == 128            # same shape


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.replica_workload("decode", 0).x_seed == 0
    assert np.isfinite(bench.max_over_ranks(float("1e-3")))
