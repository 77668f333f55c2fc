"""Host-side logic of the replica (N > 1) benchmark path, on CPU with gloo, world_size 2.

The path needs no collective: every rank runs its own replica. What the ranks
share is host logic -- the barrier around the timed region, the max over ranks
of the elapsed time, and the rule that only rank 0 prints and only rank 0 runs
the reference arm. Those are exercised here with two gloo processes.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        bench.barrier(world)
        elapsed = 10.0 + 5.0 * rank                    # per-rank timed region, ms
        mx = bench.max_over_ranks(elapsed, world, torch.device("cpu"))
        # the reference arm: ranks other than 0 exit 0 without doing any work
        ref_rc = None
        if rank != 0:
            class A:
                steps, warmup, gpus = 1, 3, world
            ref_rc = bench.run_reference(A())
        results[rank] = (mx, ref_rc)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()  # no fork of this multi-threaded process
    results = mgr.dict()
    mp.spawn(_worker, args=(world, free_port(), results), nprocs=world, join=True)
    assert results[0][0] == results[1][0] == 15.0
    assert results[1][1] == 0
