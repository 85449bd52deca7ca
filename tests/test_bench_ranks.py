"""The benchmark's multi-rank host logic on CPU: two gloo ranks take the
barrier, agree on the slowest rank's time, and report the whole-job rate of
weak-scaled replicas (the block has no exchange step, so ranks only meet
there)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    ms = 100.0 + 50.0 * rank                    # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, w)
    out[rank] = (slowest, bench.aggregate_rate(w, 32768, 10, slowest))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, rate = res[0]
    assert slowest == 150.0
    assert rate == pytest.approx(2 * 32768 * 10 / 0.150)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.aggregate_rate(1, 100, 4, 1000.0) == pytest.approx(400.0)
