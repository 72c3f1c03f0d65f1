"""The N > 1 path of bench.py on CPU: two gloo ranks (world size 2, 127.0.0.1).

The forward shards over independent heads and sequences with no exchange, so
bench.py runs one replica per rank (each with its own seed) and reduces only
the timing: the slowest rank's time, and the reference arm on rank 0 alone.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from kernelized_linear_attention_03_b300 import inputs

    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    # the slowest rank's time is the job's time
    out[rank] = bench.max_over_ranks(float(rank + 1), w)
    bench.barrier(w)
    # replicas draw different inputs (seed = rank)
    small = inputs.Workload("replica", 1, 1, 64, 16, 16, 32, "fp32", seed=rank)
    q, _, _ = inputs.make(small, "cpu")
    out[world + rank] = float(q.sum())
    # the reference arm runs on rank 0 only: other ranks return at once
    if rank != 0:
        assert bench.run_reference(None, w, rank) is None
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_reduce_the_time_and_draw_distinct_replicas():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn",
                       join=True)
    assert out[0] == out[1] == 2.0
    assert out[2] != out[3]
