"""The N > 1 host path of bench.py on CPU: two gloo ranks, each an independent
replica (no data-path collective), timed as the slowest rank, throughput summed."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [3.0, 5.0][rank]
    slow = bench.max_over_ranks(ms, world)
    rate = bench.whole_job_rate(8 * 64, slow / 1e3, world)
    out[rank] = (slow, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    world, port = 2, _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        for r in range(world):
            slow, rate = out[r]
            assert slow == 5.0
            assert rate == pytest.approx(2 * 8 * 64 / 5e-3)


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(4.5, 1) == 4.5
    assert bench.whole_job_rate(512, 0.5, 1) == 1024
