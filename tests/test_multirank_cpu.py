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


def test_bench_launcher_spawns_one_replica_per_gpu():
    # `python bench.py --gpus 2` (no WORLD_SIZE) starts two ranks itself under
    # torch.distributed.run; each derives its own device, seed and pool, and the node's
    # host memory is checked for the sum of the ranks' pools (gloo: no GPU here)
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--plan", "--workload",
                          "tiny"], cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    plans = d["plan"]
    assert [p["rank"] for p in plans] == [0, 1] and all(p["world"] == 2 for p in plans)
    assert {p["device"] for p in plans} == {"cuda:0", "cuda:1"}
    assert len({p["seed"] for p in plans}) == 2          # independent sequences per replica
    assert d["host_need_bytes"] == sum(p["host_need_bytes"] for p in plans)
    assert d["fits"] is True


def test_host_memory_check_counts_every_replica():
    import bench

    plan = {"host_need_bytes": 30 << 30}
    assert bench.host_memory_check(plan, 1, avail=40 << 30)[0]
    assert not bench.host_memory_check(plan, 1, avail=20 << 30)[0]
