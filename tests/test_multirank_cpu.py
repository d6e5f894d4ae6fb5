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


def _legs_worker(rank, world, port, out):
    """Rank 0 runs the short runs of the other configurations alone; they must not
    issue a collective the other ranks would never join."""
    import datetime
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    worlds = []

    def fake(args, w, r, local):   # what a run does with its world: a barrier and a max over ranks
        worlds.append(w)
        bench.barrier(w)
        bench.max_over_ranks(1.0, w, torch.device("cpu"))
        return {"config": {"workload": args.workload}, "run": {"launch": "direct"}, "ms_per_step": 1.0,
                "value": 1.0, "unit": "tokens/s", "kernels": {}, "clocks": None,
                "roofline": {"kernel": None, "bound": None, "frac": None, "achieved": None, "unit": None}}

    bench.native = fake
    bench.native_decode = fake
    if rank == 0:
        import argparse
        args = argparse.Namespace(workload="32k", steps=1, warmup=3)
        res = bench.other_workloads_leg(args, world, rank, 0)
        out["names"] = sorted(res)
        out["worlds"] = sorted(set(worlds))
    bench.barrier(world)
    dist.destroy_process_group()


def test_rank0_legs_issue_no_collective():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_legs_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out["names"] == ["8k", "decode", "deep", "tiny"] and out["worlds"] == [1]
