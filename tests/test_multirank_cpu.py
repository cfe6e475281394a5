"""The multi-rank parts of the benchmark on CPU, world size 2, gloo backend.

`bench.py --gpus N` runs one process per GPU: every rank times its own step
and the job's time is the slowest rank's (all-reduce MAX).  With dedicated
ownership (home page, "What DMuon Can Do": each matrix has one owner rank)
every rank must derive the same owner map and the ranks' shares must
partition the matrix set.  Both are checked here with two gloo processes.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from newton_schulz_owner_gb300 import workloads as wl
        got = bench.max_over_ranks(1.5 + rank, dist, "cpu")
        shapes = wl.WORKLOADS["llama-3.2-3b"].shapes()
        mine = bench.owned_matrices(shapes, rank, world)
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        out[rank] = (got, gathered)
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_owner_partition():
    from newton_schulz_owner_gb300 import build_lib
    if not os.path.exists(build_lib.LIB):
        build_lib.build()
    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert out[0][0] == out[1][0] == 2.5
    shares0, shares1 = out[0][1], out[1][1]
    assert shares0 == shares1                      # every rank derives the same map
    from newton_schulz_owner_gb300 import workloads as wl
    n = len(wl.WORKLOADS["llama-3.2-3b"].shapes())
    flat = sorted(i for s in shares0 for i in s)
    assert flat == list(range(n))                  # each matrix has exactly one owner
    assert abs(len(shares0[0]) - len(shares0[1])) <= n // 2
