"""The multi-GPU mode is independent replicas: check the host-side logic that
bench.py runs across ranks (rendezvous, barrier, max over ranks, whole-job
throughput) with two gloo ranks on CPU."""
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
    import bench
    r, w, _ = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    # each rank "timed" a different duration; the job time is the slowest rank's
    ms = 100.0 + 50.0 * rank
    ms_max = bench.max_over_ranks(ms, w)
    tokens_per_rank, steps = 4096, 10
    value = w * tokens_per_rank * steps / (ms_max * 1e-3)
    out[rank] = (ms_max, value)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_max_time():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:   # no fork of a multi-threaded parent
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms_max, value = res[0]
    assert ms_max == 150.0
    assert abs(value - 2 * 4096 * 10 / 0.150) < 1e-6
