"""The N > 1 host path of bench.py on CPU: two gloo ranks, each with its own
batch (weak scaling, no collective on the data path), agree on the max step
time and on the whole-job figure."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 2.0 + rank                       # rank 1 is the slow one
        ms = bench.max_over_ranks(my_ms, dist, "cpu")
        value = bench.weak_scaling_gbs(1_000_000_000, world, ms)
        dist.barrier()
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_sum_the_work():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == pytest.approx(3.0)
    assert value == pytest.approx(2 * 1e9 / 3e-3 / 1e9)


def test_single_rank_needs_no_collective():
    import bench
    assert bench.max_over_ranks(4.5) == 4.5
    assert bench.weak_scaling_gbs(6_000_000, 1, 1.0) == pytest.approx(6.0)
