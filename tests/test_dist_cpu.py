"""Multi-process host logic of bench.py on CPU (gloo, world size 2): each rank
times its own replica of the workload and rank 0 reports the slowest rank's
time; no data-path collective is involved."""
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


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, local = bench._dist()
    assert (w, r, local) == (world, rank, rank)
    # rank-dependent "timings": every rank must see the maximum
    out[rank] = bench.allreduce_max(1.5 + rank, w)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.allreduce_max(3.25, 1) == 3.25
