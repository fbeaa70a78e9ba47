"""Host-side logic of the multi-rank benchmark, on CPU with gloo (world size 2).

Each rank is an independent replica of the layer on its own token slice.  The
forward path has no collective; the bias update sums the replicas' routed counts
(one all-reduce of E int32) and applies the sign rule against the mean load of all
replicas' tokens.  The barrier and the max over ranks of the timed region give
rank 0's whole-job tokens/s.
"""
import os
import subprocess
import sys

import numpy as np
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


def _slice_logits(rank, N, E):
    """Rank r's router logits: noise plus a strong preference for expert r, so that
    each replica alone would see a different expert overloaded."""
    rng = np.random.default_rng(100 + rank)
    lg = rng.standard_normal((N, E)).astype(np.float32)
    lg[:, rank] += 3.0
    return lg


def _bias_worker(rank, world, port, q, N, E, k, step):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        idx, _ = oracle.route(_slice_logits(rank, N, E), k)
        local = oracle.dispatch(idx, E, 1)["expert_counts"]
        t = torch.from_numpy(local.copy())
        bench.counts_allreduce(world)(t).wait()
        bias0 = np.linspace(-0.05, 0.05, E, dtype=np.float32)
        glob = oracle.bias_update(t.numpy(), bias0, N * world, k, step)
        alone = oracle.bias_update(local, bias0, N, k, step)
        q.put((rank, t.numpy().tolist(), glob.tolist(), alone.tolist()))
    finally:
        dist.destroy_process_group()


def test_bias_update_over_allreduced_counts_gloo():
    """Replicas end with one bias, equal to the update of the concatenated batch;
    updating from local counts alone would have split them."""
    import oracle
    N, E, k, step = 96, 8, 2, 1e-3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 31500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_bias_worker, args=(r, 2, port, q, N, E, k, step))
             for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    lg = np.concatenate([_slice_logits(r, N, E) for r in range(2)])
    idx, _ = oracle.route(lg, k)
    counts = oracle.dispatch(idx, E, 1)["expert_counts"]
    bias0 = np.linspace(-0.05, 0.05, E, dtype=np.float32)
    want = oracle.bias_update(counts, bias0, 2 * N, k, step)
    for _, c, glob, _alone in res:
        assert c == counts.tolist()
        assert np.array_equal(np.array(glob, np.float32), want)
    assert res[0][3] != res[1][3]          # local-only updates disagree across replicas


def test_with_tokens_copies_config(moe_lib):
    from expert_routing_router_b300 import workloads as W
    c = moe_lib.config(W.DSV3_PREFILL)
    g = moe_lib.with_tokens(c, 4 * c.tokens)
    assert g.tokens == 4 * 8192 and c.tokens == 8192
    assert [getattr(g, f) for f, _ in g._fields_ if f != "tokens"] == \
        [getattr(c, f) for f, _ in c._fields_ if f != "tokens"]


def test_weak_scaling_value_single():
    assert bench.weak_scaling_value(100, 4, 1, 2.0) == 200.0


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_launch_count_per_step():
    from expert_routing_router_b300 import workloads as W
    # route: split + router GEMM + select; dispatch: count, scan, assign, permute;
    # FFN: two grouped GEMMs; combine; bias update (the launch list of the prefill layer)
    assert bench.launches_per_step(W.DSV3_PREFILL) == 11
    assert bench.launches_per_step(W.SWITCH_TOP1) == 10
    # one decode token: CUDA-core logits + select; one fused dispatch kernel + permute
    assert bench.launches_per_step(W.DSV3_DECODE.with_tokens(1)) == 8
    assert bench.launches_per_step(W.TINY_TOP2_F32) == 8


@pytest.mark.parametrize("tokens", [1, 2, 5])
def test_cpu_baseline_sample_never_exceeds_the_batch(tokens):
    """The oracle's timing sample (calibration included) stays inside the batch, down to
    a one-token decode batch."""
    from expert_routing_router_b300 import workloads as W
    w = W.Workload("decode_like", tokens, 64, 8, 2, 2, 0, 1, True, 2, 1, 0.0, 32, 16, "bf16",
                   0.0, 0.1, 1e-3)
    h = bench.oracle_inputs(W.make_inputs(w, seed=3, device="cpu"))
    import oracle
    n = bench.oracle_sample_size(oracle, w, h, budget_s=0.5)
    assert 1 <= n <= tokens
    cb = bench.cpu_baseline(w, h, budget_s=0.5)
    assert cb["value"] > 0 and f"all {tokens} tokens" in cb["sample"]
    assert f"first {n} tokens" in bench.oracle_sample_text(w, n)
    # the per-token part is scaled from the sample to the batch, the rest is not
    assert bench.oracle_rate(w, 1.0, 2.0, tokens) == tokens / 3.0


def test_clock_summary_covers_only_the_timed_region():
    """Samples taken before the timed region (the sampler's start-up, an idle GPU at its
    top clock) do not enter the median; the throttle reasons are those seen inside it."""
    import datetime
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5, 500000)

    def row(dt_ms, mhz, cap):
        ts = (t0 + datetime.timedelta(milliseconds=dt_ms)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return [ts, "0", str(mhz), "2032", "900.5", "0x4" if cap else "0x0",
                "Not Active", "Not Active", "Not Active", "Active" if cap else "Not Active"]

    rows = [row(-450, 2032, False), row(-400, 2032, False), row(-50, 2032, False),
            row(0, 1900, False), row(50, 1400, True), row(100, 1300, True)]
    c = bench.summarise_clocks(rows, t0)
    assert c["samples"] == 3 and c["sm_mhz"] == 1400.0 and c["sm_min_mhz"] == 1300.0
    assert c["sm_max_mhz"] == 2032.0 and c["reasons"] == ["sw_power_cap"]
    assert c["window"] == "timed region"
    # a region shorter than the sampling period: the sample that follows it
    c = bench.summarise_clocks(rows[:3], t0)
    assert c["samples"] == 1 and c["window"].startswith("last sample")
    assert bench.summarise_clocks([], t0)["reasons"] == ["no samples"]
