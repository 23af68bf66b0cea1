"""bench.py's multi-GPU plumbing on CPU: replicas only (no data-path
collective), a barrier around the timed region and the max over ranks.
Runs two gloo ranks on 127.0.0.1."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    ws, r, local, d = bench._dist()
    assert (ws, r, local) == (world, rank, rank)
    bench._barrier(d)
    got = bench._max_over_ranks(10.0 + rank, d)
    out[rank] = got
    d.destroy_process_group()


def test_two_gloo_replicas_take_the_max_time():
    port = 29500 + (os.getpid() % 1000)
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert dict(out) == {0: 11.0, 1: 11.0}


def test_single_process_needs_no_group():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    ws, r, local, d = bench._dist()
    assert ws == 1 and d is None
    assert bench._max_over_ranks(3.5, None) == 3.5
