"""The benchmark's multi-GPU path is replicas only (the GEMM has no exchange step): each rank
times its own copy, the job time is the slowest rank's and the work is the sum over ranks.
This checks that host-side aggregation with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    slowest = bench.max_over_ranks(dist, 1.5 + rank)          # ms per step of this replica
    total = bench.sum_over_ranks(dist, 10.0 * (rank + 1))     # work of this replica
    out[rank] = (w, r, local, slowest, total)
    dist.destroy_process_group()


def test_two_replicas_aggregate_max_time_and_summed_work():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (w, r, local, slowest, total) in res.items():
        assert (w, r, local) == (2, rank, rank)
        assert slowest == 2.5
        assert total == 30.0


def test_single_process_needs_no_process_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.0) == 3.0
    assert bench.sum_over_ranks(None, 4.0) == 4.0
