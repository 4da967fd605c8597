"""The N > 1 host path of bench.py on CPU: two gloo ranks agree on the step
count and the slowest rank's time, and the whole-job rate counts every rank's
tokens (replicas, weak scaling).  No GPU is used."""
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
        # each rank measured a different step time and chose a different count
        ms = [2.0, 3.5][rank]
        steps = [40, 25][rank]
        t, k = bench.max_over_ranks([ms * steps, steps], "cpu")
        e2e = bench.max_over_ranks([[5.0, 4.0][rank]], "cpu")[0]
        out[rank] = (t, k, e2e, bench.whole_job_rate(world, 32, t / k))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_rate():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        t, k, e2e, rate = res[r]
        assert t == 87.5 and k == 40 and e2e == 5.0     # the slowest rank, elementwise
        assert rate == pytest.approx(2 * 32 / (87.5 / 40 / 1e3))


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 7.0], "cpu") == [1.5, 7.0]
    assert bench.whole_job_rate(1, 10, 2.0) == pytest.approx(5000.0)
