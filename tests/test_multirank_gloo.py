"""Multi-rank host logic of bench.py on CPU: two gloo ranks, as torchrun
would launch them (one process per rank, 127.0.0.1 rendezvous).

The path shards with no data exchange (weak scaling: every rank quantizes
its own batch), so the only cross-rank steps are the barrier and the
max-over-ranks of the timed region; the whole-job value is the bytes of all
ranks over the slowest rank's time.
"""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_setup(world)
        dist.barrier()
        ms_local = 10.0 + 5.0 * rank           # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms_local, dist, "cpu")
        value = bench.weak_scaling_value(1e9, 10, w, ms_max)
        out[rank] = (r, w, local, ms_max, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_weak_scaling():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (r, w, local, ms_max, value) in res.items():
        assert (r, w, local) == (rank, 2, rank)
        assert ms_max == 15.0                   # the slowest rank decides
        # 2 ranks x 10 steps x 1 GB in 15 ms
        assert value == pytest.approx(2 * 10 * 1e9 / 0.015 / 1e9)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.weak_scaling_value(2e9, 5, 1, 10.0) == pytest.approx(1000.0)
