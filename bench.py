"""Benchmark of the MoE layer hot path on B300: route -> dispatch -> expert FFN -> combine
(+ selection-bias update), through the C-ABI library.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl native|reference]

One step = one pass of the whole path over one batch of seeded synthetic tokens of
the named workload (default: the DeepSeek-V3-shaped prefill layer, 8192 tokens x
7168, 256 routed experts top-8 + 1 shared, bf16).  Prints ONE JSON line on rank 0.

  value        tokens/s over all ranks, from CUDA events around each timed step on
               the launching stream (inputs resident in HBM; L2 flushed between steps
               outside the events)
  e2e          the same metric with the step's hidden states copied host->device from
               pinned memory and the layer output copied back, inside the timed region
  roofline     the expert grouped-GEMM pair (moe_expert_ffn) against measured bf16
               tensor peak; dispatch+combine against measured HBM copy bandwidth
  cpu_baseline the CPU oracle on a bounded token sample, on this host's cores
Under torchrun (N > 1) every rank runs an independent replica on its own GPU with
its own tokens (weak scaling, no collective on the data path); the time is the max
over ranks.  --impl reference times the CPU oracle (rank 0 only) on the same metric.
"""
import argparse
import datetime
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from expert_routing_router_b300 import workloads as W  # noqa: E402

L2_BYTES = 126 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="dsv3_prefill",
                    help="workload name; '<name>@<tokens>' changes the token count")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the timed backward pass (reported beside the forward metric)")
    ap.add_argument("--set", action="append", default=[], metavar="FIELD=VALUE",
                    help="override a workload field (e.g. num_experts=16), for small "
                         "profiling cases of the same kernels")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the decode sweep and the smaller layers (extra keys)")
    ap.add_argument("--no-graph", action="store_true",
                    help="issue the C-ABI calls every step instead of replaying a CUDA graph")
    return ap.parse_args()


def workload(name, overrides=()):
    import dataclasses
    base, _, n = name.partition("@")
    w = W.WORKLOADS[base]
    w = w.with_tokens(int(n)) if n else w
    for kv in overrides:
        k, _, v = kv.partition("=")
        t = type(getattr(w, k))
        w = dataclasses.replace(w, **{k: t(float(v)) if t is int else t(v)})
    if overrides:
        w = dataclasses.replace(w, name=w.name + "+" + ",".join(overrides))
    return w


def measured_ffn_traffic():
    """DRAM bytes per moe_expert_ffn call from the committed ncu launch list, if that
    capture was taken on the current kernel source (else None)."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "launches_dsv3_prefill.md")
    srcs = [os.path.join(ROOT, "expert_routing_router_b300", "csrc", f)
            for f in ("ffn_tc.cu", "tc_ptx.cuh")]
    if not os.path.exists(prof):
        return None
    vals = dict(l.split(": ", 1) for l in open(prof).read().splitlines()
                if l.startswith(("traffic_bytes_per_ffn_call:", "kernel_source_sha256_16:")))
    h = hashlib.sha256(b"".join(open(f, "rb").read() for f in srcs)).hexdigest()[:16]
    if vals.get("kernel_source_sha256_16", "").strip() != h:
        return None
    return float(vals["traffic_bytes_per_ffn_call"])


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sust=p["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sust=1400.0, src="fallback")


# ------------------------------------------------------------------ distributed plumbing
def dist_setup(gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world <= 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank, steps, world, max_seconds):
    """Whole-job tokens/s: every rank processed tokens_per_rank per step."""
    return tokens_per_rank * steps * world / max_seconds


# ------------------------------------------------------------------ clocks
class Clocks:
    """nvidia-smi sampler (every 50 ms).  It starts half a second before the timed
    region; start() marks where that region begins, and only the samples taken from
    there to stop() are summarised."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.t0 = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "50", "-i", str(index)], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        time.sleep(0.5)

    def start(self):
        self.t0 = datetime.datetime.now()

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = [r.split(", ") for r in open(self.f.name).read().strip().splitlines() if r]
        os.unlink(self.f.name)
        return summarise_clocks(rows, self.t0)


CLOCK_REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def summarise_clocks(rows, t0):
    """Median SM clock, maximum and active throttle reasons over the sampler rows taken
    at or after t0 (nvidia-smi's local timestamps, the host clock of datetime.now)."""
    def when(r):
        try:
            return datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f")
        except ValueError:
            return None
    rows = [r for r in rows if len(r) >= 10]
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    inside = [r for r in rows if t0 is not None and when(r) is not None and when(r) >= t0]
    window = "timed region"
    if not inside:  # a region shorter than the sampling period: the latest sample
        inside, window = rows[-1:], "last sample (timed region shorter than 50 ms)"
    sm = np.array([float(r[2]) for r in inside])
    reasons = sorted({CLOCK_REASONS[i] for r in inside for i in range(4)
                      if r[6 + i].strip() == "Active"})
    return {"sm_mhz": float(np.median(sm)), "sm_min_mhz": float(sm.min()),
            "sm_max_mhz": float(inside[0][3]), "reasons": reasons, "samples": len(inside),
            "window": window, "power_w_max": max(float(r[4]) for r in inside)}


# ------------------------------------------------------------------ CPU oracle
def host(t):
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_inputs(inp):
    return {k: (None if v is None else host(v)) for k, v in inp.items()}


def oracle_step(oracle, w, h, n):
    """One layer pass of the oracle on this host's cores.  Routing is per batch, so
    the router, top-k selection, dispatch tables and bias update run over all N
    tokens; the expert FFN and the combine are per token and run on the first n
    tokens (with the full batch's routing).  Returns (seconds of the full-N part,
    seconds of the n-token part)."""
    t0 = time.perf_counter()
    x = h["x"]
    logits = oracle.router_logits(x, h["w_router"], h["b_router"])
    idx, wts = oracle.route(logits, w.top_k, w.score_fn, w.normalize_topk, w.num_groups,
                            w.topk_groups, h["sel_bias"])
    d = oracle.dispatch(idx, w.num_experts, w.num_ranks, w.rank_map, w.capacity_factor,
                        w.dispatch_mode)
    t1 = time.perf_counter()
    oracle.layer_tokens(np.arange(n, dtype=np.int32), x, idx, wts, d["slot_of"],
                        h["w_gate_up"], h["w_down"], h["shared_gate_up"], h["shared_down"])
    t2 = time.perf_counter()
    if w.bias_step and h["sel_bias"] is not None:
        oracle.bias_update(d["expert_counts"], h["sel_bias"], w.tokens, w.top_k, w.bias_step)
    t3 = time.perf_counter()
    return (t1 - t0) + (t3 - t2), t2 - t1


def oracle_sample_size(oracle, w, h, budget_s):
    """Tokens of the per-token part (expert FFN + combine) that fit in about budget_s
    seconds (tokens run in parallel, so calibrate with one token per host thread)."""
    n = min(w.tokens, max(2, oracle.num_threads()))
    _, t = oracle_step(oracle, w, h, n)
    return int(max(1, min(w.tokens, budget_s / max(t / n, 1e-9))))


def oracle_rate(w, full_s, part_s, n):
    """Tokens/s of one full layer pass: the full-N part as timed, the per-token part
    scaled from n tokens to N."""
    return w.tokens / (full_s + part_s * w.tokens / n)


def oracle_sample_text(w, n):
    return (f"{w.name}: router, top-k selection, dispatch tables and bias update over all "
            f"{w.tokens} tokens; expert FFN + combine (per token) on the first {n} tokens, "
            f"time scaled by {w.tokens}/{n}; fp64 CPU oracle")


def cpu_baseline(w, h, budget_s=15.0):
    import oracle
    n = oracle_sample_size(oracle, w, h, budget_s)
    full_s, part_s = oracle_step(oracle, w, h, n)
    return {"value": oracle_rate(w, full_s, part_s, n), "unit": "tokens/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": oracle_sample_text(w, n) + f" ({full_s + part_s:.1f} s)"}


def bench_config(w, a, world, graph=True):
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": w.name, "tokens": w.tokens, "hidden": w.hidden,
            "num_experts": w.num_experts, "top_k": w.top_k, "num_ranks": w.num_ranks,
            "d_ff": w.d_ff, "shared_d_ff": w.shared_d_ff,
            "capacity_factor": w.capacity_factor, "seed": a.seed,
            "l2": "flushed between steps (252 MiB write outside the step events); "
                  "per-step working set larger than L2",
            "parallelism": f"replica x{world} (token-sharded; forward path without "
                           "collectives; with several replicas one [E] int32 all-reduce "
                           "of expert_counts feeds the bias update)",
            "launch": "one CUDA graph per C-ABI call" if graph else "direct C-ABI calls"}


# ------------------------------------------------------------------ native arm
def counts_allreduce(world):
    """Sum of the replicas' expert_counts, in place and asynchronous (the caller waits
    on the returned handle before the bias update); None on a single replica."""
    if world <= 1:
        return None
    import torch.distributed as dist
    return lambda t: dist.all_reduce(t, op=dist.ReduceOp.SUM, async_op=True)


def capture_layer(moe, b, inp, bias_step, reduce, world):
    """The layer step as CUDA graph replays.  One replica: one graph of the whole
    step.  Several: route+dispatch, expert FFN+combine and the bias update as three
    graphs, with the counts all-reduce issued eagerly between them."""
    if reduce is None:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            moe.run_layer(b, inp, bias_step=bias_step)
        return g.replay
    parts = moe.layer_parts(b, inp, bias_step, replicas=world)
    graphs = []
    for f in parts:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            f()
        graphs.append(g)

    def run():
        graphs[0].replay()
        h = reduce(b.expert_counts)
        graphs[1].replay()
        h.wait()
        graphs[2].replay()
    return run


def launches_per_step(w):
    """Kernels of this library that one forward step launches."""
    if w.act_dtype == "f32":
        n = 1                  # route: fused logits + selection
    elif w.tokens <= 16:
        n = 2                  # route: CUDA-core logits, selection
    else:
        n = 3                  # route: router weight split, tensor-core logits, selection
    one_chunk = w.tokens * w.top_k <= 2048
    n += 2 if one_chunk else 4  # dispatch: count/scan/assign (fused for one chunk), permute
    n += 2                     # expert FFN: gate_up and down grouped GEMMs
    n += 1                     # combine
    n += 1 if w.bias_step else 0
    if getattr(w, "payload", "act") == "int8":
        n += 2                 # receiver dequantisation, return-trip quantisation
    return n


def backward_launches(w):
    """Kernels of this library that one timed backward step launches (the training form:
    g, u and h saved by the forward)."""
    n = 1                      # combine backward
    n += 4                     # expert FFN backward: dgrad D1/D2, wgrad W1/W2 on the send
                               # rows (W1/W2 also write the zero gradients of empty experts)
    n += 2                     # router backward: logit gradient, dx through the router
    n += 4 if (w.act_dtype == "bf16" and w.tokens >= 128) else 1  # dW (split, GEMM, db x2)
    n += 1                     # dispatch backward
    return n


def algorithmic(w, num_kept):
    """Bytes the dispatch / combine side must move, the expert flops, and the bytes an
    all-to-all would carry, for one step."""
    s = 2 if w.act_dtype == "bf16" else 4
    N, d = w.tokens, w.hidden
    ns = N if w.shared_d_ff else 0
    flops = 6.0 * d * (w.d_ff * num_kept + w.shared_d_ff * ns)
    if getattr(w, "payload", "act") == "int8":
        q = d + 4                                            # codes + fp32 scale per row
        dispatch_bytes = N * d * s + num_kept * q            # read tokens, write codes
        dispatch_bytes += num_kept * (q + d * s)             # receiver: codes -> rows
        combine_bytes = num_kept * (d * s + q)               # expert rows -> codes
        combine_bytes += num_kept * q + (N + ns + N) * d * s  # codes + residual + shared + out
        wire = 2 * num_kept * q
    else:
        dispatch_bytes = (N + num_kept) * d * s              # read every token once, write kept rows
        combine_bytes = (num_kept + N + ns + N) * d * s      # kept rows + residual + shared + out
        wire = 2 * num_kept * d * s
    return dict(dispatch=dispatch_bytes, combine=combine_bytes, flops=flops, wire=wire)


def layer_stages(moe, b, inp, bias_step, cb):
    """(name, C-ABI call) of one layer step in path order; the INT8-payload path sends
    and returns codes.  cb: the configuration the bias update runs with."""
    c = b.cfg
    stages = [("route", lambda: moe.moe_route(c, inp["x"], inp["w_router"], inp["b_router"],
                                              inp["sel_bias"], b.logits, b.topk_idx, b.topk_w,
                                              b.workspace))]
    if b.int8_payload:
        stages += [
            ("dispatch", lambda: moe.moe_dispatch_q8(
                c, b.topk_idx, inp["x"], b.xperm_q, b.xscale, b.expert_counts, b.kept_counts,
                b.expert_start, b.rank_counts, b.rank_offsets, b.slot_of, b.perm_src,
                b.num_kept, b.workspace)),
            ("dequant", lambda: moe.moe_dequant_rows(c, b.xperm_q, b.xscale, b.perm_src,
                                                     b.xperm))]
    else:
        stages.append(("dispatch", lambda: moe.moe_dispatch(
            c, b.topk_idx, inp["x"], b.xperm, b.expert_counts, b.kept_counts, b.expert_start,
            b.rank_counts, b.rank_offsets, b.slot_of, b.perm_src, b.num_kept, b.workspace)))
    stages.append(("expert_ffn", lambda: moe.moe_expert_ffn(
        c, b.xperm, b.expert_start, b.kept_counts, inp["w_gate_up"], inp["w_down"], inp["x"],
        inp["shared_gate_up"], inp["shared_down"], b.yperm, b.yshared, b.workspace)))
    if b.int8_payload:
        stages += [
            ("quant", lambda: moe.moe_quant_rows(c, b.yperm, b.perm_src, b.yperm_q, b.yscale)),
            ("combine", lambda: moe.moe_combine_q8(c, b.yperm_q, b.yscale, b.slot_of, b.topk_w,
                                                   inp["x"], b.yshared, b.out))]
    else:
        stages.append(("combine", lambda: moe.moe_combine(c, b.yperm, b.slot_of, b.topk_w,
                                                          inp["x"], b.yshared, b.out)))
    if bias_step:
        stages.append(("bias_update", lambda: moe.moe_bias_update(cb, b.expert_counts,
                                                                  inp["sel_bias"], bias_step)))
    return stages


def time_forward(moe, w, inp, dev, flush, steps, warmup):
    """Forward layer steps of workload w on inputs inp (one CUDA graph per C-ABI call,
    CUDA events between the calls of each timed step, L2 flushed between steps outside
    the events).  Returns (per-stage mean ms, LayerBuffers after the last step)."""
    b = moe.LayerBuffers(w, device=dev)
    has_bias = bool(w.bias_step) and inp["sel_bias"] is not None
    bias0 = inp["sel_bias"].clone() if has_bias else None
    stages = layer_stages(moe, b, inp, w.bias_step if has_bias else 0.0, b.cfg)
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        for _, f in stages:
            f()
    torch.cuda.synchronize()
    runs = []
    for _, f in stages:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            f()
        runs.append(g.replay)
    for _ in range(warmup):
        for r in runs:
            r()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(runs) + 1)]
           for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.fill_(i & 0xff)
        evs[i][0].record(s)
        for j, r in enumerate(runs):
            r()
            evs[i][j + 1].record(s)
    torch.cuda.synchronize()
    per = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(len(runs))] for e in evs])
    if has_bias:
        inp["sel_bias"].copy_(bias0)
    assert int(b.workspace[:4].view(torch.int32).item()) == 0, "device status word set"
    return {n: float(v) for (n, _), v in zip(stages, per.mean(axis=0))}, b


def sweep(a, moe, inp, dev, flush, pk):
    """The other workloads, forward only, each on one GPU: the DeepSeek-V3 decode sweep
    (the prefill layer's weights, fresh tokens at every batch size) with its expert
    weight stream against the HBM peak, then the smaller layers."""
    steps, warmup = 20, 5
    out = {"decode": {}, "layers": {}}
    s_b = 2
    for T in W.DECODE_TOKENS:
        w = W.DSV3_DECODE.with_tokens(T)
        inp_t = dict(inp, x=W.make_tokens(w, T, seed=a.seed, device=dev))
        st, b = time_forward(moe, w, inp_t, dev, flush, steps, warmup)
        ms = sum(st.values())
        touched = int((b.kept_counts > 0).sum().item())
        wbytes = (touched * 3 * w.hidden * w.d_ff + 3 * w.hidden * w.shared_d_ff) * s_b
        ffn_gbs = wbytes / (st["expert_ffn"] * 1e-3) / 1e9
        out["decode"][str(T)] = {
            "tokens_per_s": T / (ms * 1e-3), "ms_per_step": ms,
            "stage_ms": st, "experts_touched": touched,
            "expert_weight_bytes_per_step": wbytes,
            "expert_ffn_weight_gbs": ffn_gbs, "expert_ffn_frac_of_hbm": ffn_gbs / pk["hbm"],
            "step_weight_gbs": wbytes / (ms * 1e-3) / 1e9,
            "step_frac_of_hbm": wbytes / (ms * 1e-3) / 1e9 / pk["hbm"]}
        del b
    for name in ("tiny_top2_f32", "switch_top1_bf16", "gshard_top2_skewed",
                 "gshard_top2_padded", "dsv3_prefill_int8"):
        w = W.WORKLOADS[name]
        # the INT8-payload layer has the prefill layer's draws: reuse its inputs
        inp_w = inp if name == "dsv3_prefill_int8" else W.make_inputs(w, seed=a.seed,
                                                                      device=dev)
        st, b = time_forward(moe, w, inp_w, dev, flush, steps, warmup)
        ms = sum(st.values())
        nk = int(b.num_kept.item())
        alg = algorithmic(w, nk)
        dc_ms = sum(v for n, v in st.items() if n in ("dispatch", "dequant", "quant", "combine"))
        ffn_tf = alg["flops"] / (st["expert_ffn"] * 1e-3) / 1e12
        out["layers"][name] = {
            "tokens_per_s": w.tokens / (ms * 1e-3), "ms_per_step": ms, "stage_ms": st,
            "dtype": "f32" if w.act_dtype == "f32" else "bf16",
            "drop_rate": 1.0 - nk / (w.tokens * w.top_k),
            "expert_ffn_tflops": ffn_tf,
            "expert_ffn_frac_of_bf16_peak": (ffn_tf / pk["bf16"]) if w.act_dtype == "bf16"
                                            else None,
            "dispatch_combine_gbs": (alg["dispatch"] + alg["combine"]) / (dc_ms * 1e-3) / 1e9}
        del b
        if inp_w is not inp:
            del inp_w
        torch.cuda.empty_cache()
    out["note"] = ("forward only, 20 timed steps after 5 warm-up steps each, one CUDA graph "
                   "per C-ABI call, L2 flushed between steps; decode weight bytes = (experts "
                   "that received rows + the shared expert) x 3 d F x 2 B")
    return out


def run_native(a, w, rank, world, local):
    from expert_routing_router_b300 import moe
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    # every replica holds the same layer (weights, router, selection bias) and its own
    # token batch
    inp = W.make_inputs(w, seed=a.seed, device=dev)
    if rank > 0:
        inp["x"] = W.make_tokens(w, w.tokens, seed=a.seed + rank, device=dev)
    b = moe.LayerBuffers(w, device=dev)
    step_bias = w.bias_step
    bias0 = None if inp["sel_bias"] is None else inp["sel_bias"].clone()
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream()

    c = b.cfg
    has_bias = bool(step_bias) and inp["sel_bias"] is not None
    # the bias update applies the sign rule to the routed counts of all replicas
    reduce = counts_allreduce(world) if has_bias else None
    cb = moe.with_tokens(c, w.tokens * world) if world > 1 else c
    stages = layer_stages(moe, b, inp, step_bias if has_bias else 0.0, cb)
    names = [n for n, _ in stages]
    n_st = len(stages)

    def step(runs, evs=None):
        h = None
        if evs is not None:
            evs[0].record(s)
        for j, r in enumerate(runs):
            if names[j] == "bias_update" and h is not None:
                h.wait()              # the summed counts feed the bias update
            r()
            if names[j] == "dispatch" and reduce is not None:
                h = reduce(b.expert_counts)   # overlaps the expert FFN and combine
            if evs is not None:
                evs[j + 1].record(s)

    calls = [f for _, f in stages]
    for _ in range(a.warmup):
        step(calls)
    torch.cuda.synchronize()
    if bias0 is not None:
        inp["sel_bias"].copy_(bias0)
    assert int(b.workspace[:4].view(torch.int32).item()) == 0, "device status word set"
    num_kept = int(b.num_kept.item())

    # each C-ABI call captured as its own CUDA graph, so that events between the graph
    # launches time every stage inside the timed region
    runs = calls
    if not a.no_graph:
        runs = []
        for f in calls:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                f()
            runs.append(g.replay)
        torch.cuda.synchronize()
        for _ in range(a.warmup):
            step(runs)
        torch.cuda.synchronize()
        if bias0 is not None:
            inp["sel_bias"].copy_(bias0)

    # ---------------- timed: K steps; CUDA events between the C-ABI calls of every step,
    # on the launching stream
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_st + 1)]
           for _ in range(a.steps)]
    clk = Clocks(dev.index) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    if clk:
        clk.start()
    for i in range(a.steps):
        flush.fill_(i & 0xff)            # L2 flush, outside the step's events
        step(runs, evs[i])
    torch.cuda.synchronize()
    barrier(world)
    per = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(n_st)] for e in evs])  # ms
    step_ms = per.sum(axis=1)
    total_s = max_over_ranks(step_ms.sum() / 1e3, world)
    value = weak_scaling_value(w.tokens, a.steps, world, total_s)
    stage_ms = {n: float(v) for n, v in zip(names, per.mean(axis=0))}
    ffn_ms = stage_ms["expert_ffn"]
    # every stage on the dispatch / combine side of the expert FFN
    dc_ms = sum(v for n, v in stage_ms.items() if n in ("dispatch", "dequant", "quant", "combine"))
    status = int(b.workspace[:4].view(torch.int32).item())
    if bias0 is not None:
        inp["sel_bias"].copy_(bias0)

    # ---------------- end to end through the C ABI with host buffers
    # Every step copies its own hidden states host->device (pinned) and its layer
    # output device->host inside the timed region.  Two buffer sets, each with its own
    # captured graph, let the copies of neighbouring steps run on a copy stream while
    # a step computes (as a serving loop would); nothing is reused across steps.
    io_bytes = w.tokens * w.hidden * (2 if w.act_dtype == "bf16" else 4)
    x_host = [torch.empty(w.tokens, w.hidden, dtype=w.torch_dtype, pin_memory=True)
              for _ in range(2)]
    for xh in x_host:
        xh.copy_(inp["x"])
    out_host = [torch.empty_like(x_host[0], pin_memory=True) for _ in range(2)]
    sets = []
    for i in range(2):
        xi = inp["x"] if i == 0 else inp["x"].clone()
        bi = b if i == 0 else moe.LayerBuffers(w, device=dev)
        inp_i = dict(inp, x=xi)

        def step_i(bb=bi, ii=inp_i):
            moe.run_layer(bb, ii, bias_step=step_bias, reduce_counts=reduce, replicas=world)
        run_i = step_i
        if not a.no_graph:
            step_i()
            torch.cuda.synchronize()
            run_i = capture_layer(moe, bi, inp_i, step_bias, reduce, world)
        sets.append((xi, bi, run_i))
    if bias0 is not None:
        inp["sel_bias"].copy_(bias0)
    # compute and copies on two streams of their own (the legacy default stream would
    # serialise with the copy stream)
    copy_s = torch.cuda.Stream(device=dev)   # host -> device
    back_s = torch.cuda.Stream(device=dev)   # device -> host (the link is full duplex)
    comp_s = torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s = comp_s
    torch.cuda.set_stream(comp_s)
    e0.record(s)
    for i in range(a.steps):
        j = i & 1
        xi, bi, run_i = sets[j]
        with torch.cuda.stream(copy_s):
            if i >= 2:
                copy_s.wait_event(comp_done[j])   # step i-2 no longer reads this x
            xi.copy_(x_host[j], non_blocking=True)
            h2d_done[j].record(copy_s)
        s.wait_event(h2d_done[j])
        if i >= 2:
            s.wait_event(d2h_done[j])             # step i-2's output has left this buffer
        run_i()
        comp_done[j].record(s)
        with torch.cuda.stream(back_s):
            back_s.wait_event(comp_done[j])
            out_host[j].copy_(bi.out, non_blocking=True)
            d2h_done[j].record(back_s)
    s.wait_stream(copy_s)
    s.wait_stream(back_s)
    e1.record(s)
    torch.cuda.synchronize()
    torch.cuda.set_stream(torch.cuda.default_stream(dev))
    barrier(world)
    clocks = clk.stop() if clk else None  # sampled over the timed and e2e loops
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    e2e_value = weak_scaling_value(w.tokens, a.steps, world, e2e_s)
    if bias0 is not None:
        inp["sel_bias"].copy_(bias0)
    del sets

    # ---------------- roofline figures
    pk = peaks()
    alg = algorithmic(w, num_kept)
    flops = alg["flops"]
    ffn_tflops = flops / (ffn_ms * 1e-3) / 1e12
    # dispatch+combine: bytes over the time of every call on that side; the dispatch
    # call also holds the count / scan / assign kernels, included here (conservative)
    dc_gbs = (alg["dispatch"] + alg["combine"]) / (dc_ms * 1e-3) / 1e9
    out = {
        "metric": "MoE-layer tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": float(step_ms.mean()),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.act_dtype == "bf16" else "f32", "data": "synthetic",
        "config": bench_config(w, a, world, graph=not a.no_graph),
        "roofline": {"kernel": "expert grouped GEMMs (gate_up+SwiGLU, down) of moe_expert_ffn",
                     "bound": "tensor", "achieved": ffn_tflops, "peak": pk["bf16"],
                     "unit": "TFLOP/s", "frac": ffn_tflops / pk["bf16"],
                     "peak_kind": f"{pk['src']} burst bf16 (the 1.1 kW power cap engages "
                                  "after about six back-to-back steps and slows the later "
                                  "ones; frac_of_sustained is against the capped figure; "
                                  "see clocks)",
                     "frac_of_sustained": ffn_tflops / pk["bf16_sust"],
                     "traffic": (measured_ffn_traffic() if w.name == "dsv3_prefill" else None),
                     "traffic_unit": "bytes per moe_expert_ffn call (ncu dram read+write)",
                     "algorithmic_flops_per_launch": flops},
        "dispatch_combine": {"bytes": alg["dispatch"] + alg["combine"], "achieved": dc_gbs,
                             "unit": "GB/s", "peak": pk["hbm"], "frac": dc_gbs / pk["hbm"],
                             "frac_of_8TBs": dc_gbs / 8000.0,
                             "payload": getattr(w, "payload", "act"),
                             "all_to_all_bytes_per_step": alg["wire"]},
        "stage_ms": dict(stage_ms, note="events between the calls of each timed step"),
        "routing": {"num_kept": num_kept, "drop_rate": 1.0 - num_kept / (w.tokens * w.top_k)},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": io_bytes,
                "d2h_bytes_per_step": io_bytes,
                "how": "pinned host x -> device and layer output -> host every step, on two copy "
                       "streams overlapping the neighbouring steps (two buffer sets)"},
        "clocks": clocks, "gpu_launches": launches_per_step(w) * a.steps,
        "device_status": status,
    }
    if (not a.no_backward and w.act_dtype == "bf16" and getattr(w, "payload", "act") == "act"
            and world == 1):
        out["backward"] = time_backward(a, w, moe, b, inp, s, flush, pk)
        # training step = the forward with its expert FFN in the saving form + backward
        fwd_bwd_ms = (out["ms_per_step"] - stage_ms["expert_ffn"] +
                      out["backward"]["expert_ffn_save_ms"] + out["backward"]["ms_per_step"])
        out["backward"]["train_step_tokens_per_s"] = w.tokens / (fwd_bwd_ms * 1e-3)
    if (not a.no_sweep and world == 1 and w.name == "dsv3_prefill"):
        out["sweep"] = sweep(a, moe, inp, dev, flush, pk)
    if getattr(w, "payload", "act") == "int8":
        out["cpu_baseline"] = None           # the oracle baseline times the bf16-payload layer
    elif rank == 0 and world == 1 and not a.no_cpu_baseline:
        del b, flush
        torch.cuda.empty_cache()
        out["cpu_baseline"] = cpu_baseline(w, oracle_inputs(inp))
    return out


def time_backward(a, w, moe, b, inp, s, flush, pk):
    """The layer's backward calls on the forward state held in b, timed like the
    forward: one CUDA graph per call, events between the calls of each timed step,
    L2 flushed between steps.  Reported beside the forward metric."""
    dev = b.logits.device
    s = torch.cuda.current_stream()      # the stream the calls below launch on
    g = moe.GradBuffers(w, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(a.seed + 1000)
    dout = torch.randn(w.tokens, w.hidden, generator=gen, device=dev).to(w.torch_dtype)
    c = b.cfg
    # the training forward keeps h and g|u for the backward (moe_expert_ffn_save); time
    # its expert-FFN call against the inference one it replaces
    saved = torch.empty(moe.moe_saved_size(c), dtype=torch.uint8, device=dev)

    def ffn_save():
        moe.moe_expert_ffn_save(c, b.xperm, b.expert_start, b.kept_counts, inp["w_gate_up"],
                                inp["w_down"], inp["x"], inp["shared_gate_up"],
                                inp["shared_down"], b.yperm, b.yshared, saved, b.workspace)
    for _ in range(a.warmup):
        ffn_save()
    save_ms = []
    for i in range(a.steps):
        flush.fill_(i & 0xff)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        ffn_save()
        e1.record(s)
        torch.cuda.synchronize()
        save_ms.append(e0.elapsed_time(e1))
    save_ms = float(np.mean(save_ms))
    calls = [
        ("combine_bwd", lambda: moe.moe_combine_backward(c, dout, b.yperm, b.slot_of, b.topk_w,
                                                         g.dyperm, g.dtopk_w)),
        ("expert_ffn_bwd", lambda: moe.moe_expert_ffn_backward(
            c, b.xperm, b.expert_start, b.kept_counts, inp["w_gate_up"], inp["w_down"],
            inp["x"], inp["shared_gate_up"], inp["shared_down"], g.dyperm, dout, g.dxperm,
            g.dx_shared, g.dw_gate_up, g.dw_down, g.dshared_gate_up, g.dshared_down,
            g.workspace, saved=saved)),
        ("route_bwd", lambda: moe.moe_route_backward(c, inp["x"], inp["w_router"], b.logits,
                                                     b.topk_idx, g.dtopk_w, g.dlogits,
                                                     g.dx_router, g.dw_router, g.db_router,
                                                     g.workspace)),
        ("dispatch_bwd", lambda: moe.moe_dispatch_backward(c, g.dxperm, b.slot_of, dout,
                                                           g.dx_shared, g.dx_router, g.dx)),
    ]
    for _ in range(a.warmup):
        for _, f in calls:
            f()
    torch.cuda.synchronize()
    runs = [f for _, f in calls]
    if not a.no_graph:
        runs = []
        for _, f in calls:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                f()
            runs.append(gr.replay)
        for _ in range(a.warmup):
            for r in runs:
                r()
        torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(runs) + 1)]
           for _ in range(a.steps)]
    clk = Clocks(dev.index)
    torch.cuda.synchronize()
    clk.start()
    for i in range(a.steps):
        flush.fill_(i & 0xff)
        evs[i][0].record(s)
        for j, r in enumerate(runs):
            r()
            evs[i][j + 1].record(s)
    torch.cuda.synchronize()
    clocks = clk.stop()
    per = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(len(runs))] for e in evs])
    stage = {n: float(v) for (n, _), v in zip(calls, per.mean(axis=0))}
    step_ms = float(per.sum(axis=1).mean())
    status = int(g.workspace[:4].view(torch.int32).item())
    nk = int(b.num_kept.item())
    rows_f = w.d_ff * nk + w.shared_d_ff * (w.tokens if w.shared_d_ff else 0)
    alg = 12.0 * w.hidden * rows_f      # dgrad (2 GEMMs) + wgrad (2 GEMMs)
    t = stage["expert_ffn_bwd"] * 1e-3
    del g, saved
    return {"metric": "MoE-layer backward tokens/s", "value": w.tokens / (step_ms * 1e-3),
            "unit": "tokens/s", "ms_per_step": step_ms,
            "train_step_tokens_per_s": None,
            "stage_ms": dict(stage, note="events between the calls of each timed step"),
            "expert_ffn_bwd": {"bound": "tensor", "unit": "TFLOP/s",
                               "achieved": alg / t / 1e12,
                               "peak": pk["bf16"], "frac": alg / t / 1e12 / pk["bf16"],
                               "algorithmic_flops": alg,
                               "note": "dgrad + wgrad, 12 d F flops per row; h and g|u come "
                                       "from the training forward (moe_expert_ffn_save)"},
            "expert_ffn_save_ms": save_ms,
            "clocks": clocks, "gpu_launches": backward_launches(w) * a.steps, "device_status": status}


# ------------------------------------------------------------------ reference arm
def run_reference(a, w):
    """The CPU oracle as it stands, on this host's cores: same workload, config, metric
    and unit as the native arm; each step is one layer pass with the per-token part on
    a bounded sample (oracle_step)."""
    import oracle
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    h = oracle_inputs(W.make_inputs(w, seed=a.seed, device=dev))
    steps = max(1, a.steps + a.warmup)
    full_s, _ = oracle_step(oracle, w, h, 1)
    budget = max(0.5, 120.0 / steps - full_s)
    n = oracle_sample_size(oracle, w, h, budget)
    for _ in range(a.warmup):
        oracle_step(oracle, w, h, n)
    full, part = 0.0, 0.0
    for _ in range(a.steps):
        f, p = oracle_step(oracle, w, h, n)
        full, part = full + f, part + p
    value = oracle_rate(w, full, part, n)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return {"impl": "reference", "metric": "MoE-layer tokens/s", "value": value,
            "unit": "tokens/s", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": w.tokens / value * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(w, a, world, graph=not a.no_graph),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": "each step: " + oracle_sample_text(w, n)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    a = parse()
    w = workload(a.config, a.set)
    if a.impl == "reference":
        # rank 0 alone times the CPU oracle; other ranks exit without work
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(run_reference(a, w)), flush=True)
        return
    rank, world, local = dist_setup(a.gpus)
    out = run_native(a, w, rank, world, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
