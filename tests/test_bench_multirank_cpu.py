"""Host-side logic of the multi-rank benchmark, on CPU with gloo (world size 2).

Each rank is an independent replica on its own token slice (no collective on the
data path); the only cross-rank steps are the barrier and the max over ranks of the
timed region, from which rank 0 reports whole-job tokens/s.
"""
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        seconds = [1.5, 2.0][rank]                      # rank 1 is the slow one
        t = bench.max_over_ranks(seconds, world)
        v = bench.weak_scaling_value(8192, 10, world, t)
        q.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]            # both ranks see the max
    assert res[0][2] == pytest.approx(8192 * 10 * 2 / 2.0)


def test_weak_scaling_value_single():
    assert bench.weak_scaling_value(100, 4, 1, 2.0) == 200.0


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_launch_count_per_step():
    from expert_routing_router_b300 import workloads as W
    assert bench.launches_per_step(W.DSV3_PREFILL) == 9
    assert bench.launches_per_step(W.SWITCH_TOP1) == 8
