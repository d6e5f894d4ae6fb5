"""Replica timing across ranks, on the CPU with gloo (world size 2).

The lazy step shards by sequence with no collective on the data path; the
only cross-rank operations are the barrier around the timed region and the
max over ranks of the elapsed time, both exercised here."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, l = bench.dist_info()
    assert (w, r, l) == (world, rank, rank)
    dist = bench.dist_init(world, "gloo")
    bench.barrier(world)
    elapsed = 1.5 + rank                       # rank 1 is the slower replica
    t = bench.max_over_ranks(elapsed, world, torch.device("cpu"))
    out[rank] = t
    # the reference arm runs on rank 0 only
    import argparse
    args = argparse.Namespace(workload="tiny", steps=1, warmup=3, ref_budget=1.0)
    if rank != 0:
        assert bench.reference(args, world, rank) is None
    bench.barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_with_gloo():
    world = 2
    # the result dict's server process is spawned too: forking a process whose
    # earlier tests left worker threads running can deadlock the child
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == 2.5
