"""The multi-rank path of bench.py on CPU: two gloo ranks.

With N ranks every rank runs its own replica of the workload (weak scaling,
no collective on the data path); the only cross-rank operations are the
barrier around the timed region and the max-over-ranks of the timings,
which these tests exercise with the gloo backend.
"""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    t = bench.max_over_ranks(10.0 * rank + 1.5, ws)
    results[rank] = t
    bench.barrier(ws)
    dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(2, port, results), nprocs=2, join=True, start_method="spawn")
        assert dict(results) == {0: 11.5, 1: 11.5}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)   # no-op without a process group
