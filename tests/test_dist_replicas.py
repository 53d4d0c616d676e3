"""The benchmark's several-GPU host logic on CPU, with two gloo ranks.

The path shards into independent replicas (each rank packs and receives its
own batch, no data-path collective), so what several processes add is host
logic only: each rank's own batch, the time taken as the slowest rank's, the
tokens of all ranks counted in the value, and the reference arm run by rank 0
alone.  These run as two real processes over gloo on 127.0.0.1.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # the slowest rank's time, on every rank
        t = bench.max_over_ranks(dist, 10.0 + 5.0 * rank, "cpu")
        # each rank's own batch of the same shape
        w = workloads.make(1, T=64, H=256, **bench.replica_workload_kwargs(rank, 1))
        digest = float(np.asarray(w.tokens, np.float64).sum())
        # the reference arm: rank 0 only
        args = type("A", (), {"steps": 1, "warmup": 0, "config": 1})()
        ref_none = bench.reference_arm(args, rank, world) is None if rank else None
        out[rank] = (t, w.tokens.shape, w.topk.shape, digest, ref_none)
    finally:
        dist.destroy_process_group()


def test_two_replicas_over_gloo():
    world = 2
    with mp.get_context("spawn").Manager() as m:   # no fork of this (multi-threaded) process
        out = m.dict()
        mp.spawn(rank_main, args=(world, free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0          # max over ranks on both
    assert res[0][1] == res[1][1] and res[0][2] == res[1][2]
    assert res[0][3] != res[1][3]                  # different data per replica
    assert res[1][4] is True                       # rank 1 does not run the reference arm


def test_one_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(None, 3.5, "cpu") == 3.5
    assert bench.replica_workload_kwargs(0) == {}
    assert bench.replica_workload_kwargs(3, 2) == {"seed": 3002}
    # the default workload is the largest configuration (seed 4)
    assert bench.replica_workload_kwargs(3) == {"seed": 3004}
