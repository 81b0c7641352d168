"""The benchmark's whole-job aggregation over ranks (max of the per-rank
times, sum of the per-rank iterations), run as two gloo ranks on CPU."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, iters = bench.aggregate(10.0 * (rank + 1), 100 * (rank + 1), world, "cpu")
        out[rank] = (ms, iters)
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    # every rank sees the slowest rank's time and all ranks' iterations
    assert res == {0: (20.0, 300), 1: (20.0, 300)}


def test_aggregate_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(12.5, 77, 1, "cpu") == (12.5, 77)
