"""The multi-GPU path is replicas only (the linear layer needs no exchange
between GPUs): bench.py's ranks meet at a barrier around the timed region and
report the slowest rank's time.  This runs that plumbing as two gloo ranks on
the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    r, w, local = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    try:
        bench.barrier(dist)
        # each rank's "time": the slowest one is what the job reports
        t = bench.max_over_ranks(dist, 1.5 + r, torch.device("cpu"))
        bench.barrier(dist)
        out[rank] = (r, w, local, t)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        assert dict(out) == {0: (0, 2, 0, 2.5), 1: (1, 2, 1, 2.5)}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.0, torch.device("cpu")) == 3.0
