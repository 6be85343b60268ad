"""Multi-GPU runs of the step are independent replicas (sequences never cross ranks, so there
is no collective on the data path).  The only cross-rank logic is the benchmark's barrier and
max-over-ranks timing, tested here with two gloo ranks on CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    d = bench.dist_init(w, "gloo")
    bench.barrier(d, torch.device("cpu"))
    # each replica measured its own step time; the job's time is the slowest rank's
    t = bench.max_over_ranks(1.0 + rank, d, torch.device("cpu"))
    results[rank] = t
    d.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_replicas_report_the_slowest_rank():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this multi-threaded process
        results = m.dict()
        mp.spawn(_worker, args=(2, port, results), nprocs=2, join=True)
        assert dict(results) == {0: 2.0, 1: 2.0}


def test_single_process_needs_no_process_group():
    assert bench.dist_init(1, "gloo") is None
    assert bench.max_over_ranks(3.5, None, torch.device("cpu")) == 3.5
