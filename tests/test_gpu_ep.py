"""Expert-parallel layer on one GPU: every rank's route, dispatch, local experts,
shared expert and combine run through the C ABI, the exchanges as copies between the
ranks' buffers (ranks one after another; no rank waits on another).  Each rank's
layer is checked against the oracle step by step, exactly as a single-device layer
on that rank's tokens, with the expert FFN rows computed on the rank that owns the
expert and brought back by the return exchange.
"""
import dataclasses

import numpy as np
import pytest
import torch

from expert_routing_router_b300 import ep, workloads as W
from test_gpu_parity import check_layer, host, host_weights, small

pytestmark = pytest.mark.gpu


def _ranks(w, R, seed=0, **kw):
    """R ranks of the layer: the same weights, each its own slice of the tokens."""
    whole = W.make_inputs(dataclasses.replace(w, tokens=w.tokens * R), seed=seed, device="cuda")
    ranks = []
    for r in range(R):
        inp = dict(whole)
        inp["x"] = whole["x"][r * w.tokens:(r + 1) * w.tokens].contiguous()
        ranks.append(ep.RankLayer(w, r, inp, **kw))
    return ranks, whole


EP_CASES = {
    # 2 ranks, contiguous experts, sigmoid + groups, shared expert, no capacity
    "two_ranks_contiguous_shared": (small(tokens=600, hidden=264, num_experts=16, top_k=4,
                                          num_ranks=2, d_ff=200, shared_d_ff=72), 2),
    # 4 ranks, round-robin experts, softmax, capacity with drops
    "four_ranks_round_robin_capacity": (small(tokens=300, hidden=136, num_experts=10, top_k=3,
                                              num_ranks=4, rank_map=1, score_fn=0,
                                              num_groups=1, topk_groups=1, capacity_factor=1.0,
                                              d_ff=96, shared_d_ff=0, sel_bias_std=0.0), 4),
    # few rows per expert: the token-major small-segment kernels (local experts and the
    # shared-expert call with no routed rows)
    "decode_sized_two_ranks": (small(tokens=40, hidden=264, num_experts=64, top_k=4,
                                     num_ranks=2, num_groups=8, topk_groups=4, d_ff=200,
                                     shared_d_ff=72), 2),
    # many rows per expert: the SM-pair kernels on both sides
    "pair_kernel_two_ranks": (small(tokens=1500, hidden=264, num_experts=4, top_k=2,
                                    num_ranks=2, num_groups=2, topk_groups=1, d_ff=200,
                                    shared_d_ff=72), 2),
    # DeepSeek-V3-shaped experts on 2 ranks (128 local experts each), fewer tokens
    "dsv3_shape_two_ranks": (dataclasses.replace(W.DSV3_PREFILL, name="dsv3_ep", tokens=1024,
                                                 num_ranks=2), 2),
}


@pytest.mark.parametrize("name", list(EP_CASES))
def test_expert_parallel_layer_loopback(name):
    w, R = EP_CASES[name]
    ranks, whole = _ranks(w, R)
    sb0 = None if whole["sel_bias"] is None else whole["sel_bias"].clone()
    plans = ep.run_layer_loopback(ranks, bias_step=w.bias_step)
    torch.cuda.synchronize()
    hw = host_weights(whole)
    total = 0
    for r, (rank, plan) in enumerate(zip(ranks, plans)):
        assert int(rank.b.workspace[:4].view(torch.int32).item()) == 0
        assert int(rank.local_ws[:4].view(torch.int32).item()) == 0
        # the plan's send chunks are this rank's dispatch segments
        st = host(rank.b.expert_start)
        for (dst, e, off, n) in plan.send_chunks:
            assert off == st[e]
        total += plan.recv_rows
        if sb0 is not None:  # check this rank's layer with the bias it routed with
            rank.inp = dict(rank.inp, sel_bias=sb0)
        n_tok = None if w.tokens <= 1024 and w.hidden <= 1024 else 96
        check_layer(w, rank.inp, rank.b, n_sample_tokens=n_tok,
                    n_sample_rows=None if n_tok is None else 256, seed=r, hw=hw)
    assert total == sum(int(rk.b.num_kept.item()) for rk in ranks)
    if sb0 is not None and w.bias_step:
        # sign rule on the counts summed over the ranks (all ranks' tokens)
        counts = sum(host(rk.b.expert_counts).astype(np.int64) for rk in ranks)
        mean_num = w.tokens * R * w.top_k
        sgn = np.sign(counts * w.num_experts - mean_num)
        ref = (host(sb0) - np.float32(w.bias_step) * sgn.astype(np.float32)).astype(np.float32)
        np.testing.assert_array_equal(host(whole["sel_bias"]), ref)


def test_expert_parallel_layer_dist_single_rank():
    """run_layer_dist through an NCCL process group of one rank: the all-gather of the
    kept counts, the plan, both exchanges (all chunks are this rank's own), the local
    experts, the shared expert, the combine and the all-reduced bias update."""
    import os
    import socket
    import torch.distributed as dist
    w, _ = EP_CASES["two_ranks_contiguous_shared"]
    w = dataclasses.replace(w, num_ranks=1)
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                            world_size=1)
    try:
        ranks, whole = _ranks(w, 1, seed=4)
        sb0 = whole["sel_bias"].clone()
        plan = ep.run_layer_dist(ranks[0], bias_step=w.bias_step)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    r = ranks[0]
    assert plan.recv_rows == int(r.b.num_kept.item())
    assert int(r.local_ws[:4].view(torch.int32).item()) == 0
    check_layer(w, dict(r.inp, sel_bias=sb0), r.b)
    counts = host(r.b.expert_counts).astype(np.int64)
    sgn = np.sign(counts * w.num_experts - w.tokens * w.top_k)
    ref = (host(sb0) - np.float32(w.bias_step) * sgn.astype(np.float32)).astype(np.float32)
    np.testing.assert_array_equal(host(whole["sel_bias"]), ref)


def test_expert_parallel_int8_payload_matches_the_single_device_layer():
    """INT8 codes + scales cross both exchanges (dispatch_q8 on the source, dequant and
    quant around the local experts, combine_q8 back home).  Each rank's layer is compared
    with the single-device INT8 layer on the same tokens: the routing, the send codes
    and scales bit for bit, and the output within the bf16 layer tolerance (the expert
    rows are the same products in the same order, grouped into other tiles)."""
    from expert_routing_router_b300 import moe
    w = small(tokens=300, hidden=264, num_experts=16, top_k=4, num_ranks=2, d_ff=200,
              shared_d_ff=72, bias_step=0.0, payload="int8")
    ranks, whole = _ranks(w, 2, seed=6)
    ep.run_layer_loopback(ranks)
    torch.cuda.synchronize()
    for r, rank in enumerate(ranks):
        assert int(rank.b.workspace[:4].view(torch.int32).item()) == 0
        one = moe.LayerBuffers(w)
        moe.run_layer(one, rank.inp)
        torch.cuda.synchronize()
        for name in ("topk_idx", "slot_of", "perm_src", "kept_counts"):
            np.testing.assert_array_equal(host(getattr(rank.b, name)), host(getattr(one, name)),
                                          err_msg=name)
        kept = np.nonzero(host(one.perm_src) >= 0)[0]
        rows = torch.from_numpy(kept).cuda().long()
        np.testing.assert_array_equal(host(rank.b.xperm_q[rows]), host(one.xperm_q[rows]))
        np.testing.assert_array_equal(host(rank.b.xscale[rows]), host(one.xscale[rows]))
        got = rank.b.out.double().cpu().numpy()
        ref = one.out.double().cpu().numpy()
        x = rank.inp["x"].double().cpu().numpy()
        # the MoE part (out - x) within 2e-2 of its own scale, plus the storage rounding of
        # out, so that an error in the exchanged expert rows cannot hide behind the residual
        allow = 2e-2 * np.max(np.abs(ref - x)) + 2.0 ** -8 * np.abs(ref)
        assert np.all(np.abs((got - x) - (ref - x)) <= allow)


# ---------------------------------------------------------------- overlapped schedule

OVERLAP_CASES = {
    # (workload, ranks, source groups, fixed plan on a capacity-padded send buffer)
    "two_ranks_two_groups": (EP_CASES["two_ranks_contiguous_shared"][0], 2, 2, False),
    "four_ranks_two_groups_round_robin_capacity":
        (EP_CASES["four_ranks_round_robin_capacity"][0], 4, 2, False),
    "four_ranks_four_groups_static": (small(tokens=300, hidden=136, num_experts=12, top_k=3,
                                            num_ranks=4, rank_map=1, score_fn=0, num_groups=1,
                                            topk_groups=1, capacity_factor=1.0, d_ff=96,
                                            shared_d_ff=64, sel_bias_std=0.0,
                                            dispatch_mode=1), 4, 4, True),
    "two_ranks_static_int8": (small(tokens=300, hidden=264, num_experts=16, top_k=4,
                                    num_ranks=2, capacity_factor=1.1, d_ff=200, shared_d_ff=72,
                                    dispatch_mode=1, payload="int8"), 2, 2, True),
    "dsv3_shape_two_ranks_two_groups": (EP_CASES["dsv3_shape_two_ranks"][0], 2, 2, False),
}


@pytest.mark.parametrize("name", list(OVERLAP_CASES))
def test_expert_parallel_overlapped_schedule(name):
    """The exchange and the local experts in steps over source groups, the copies on a
    second stream (group g's expert FFN waits only for group g's rows; results go back
    while the next group computes).  Each rank's layer is checked against the oracle,
    and against the same rank's tokens as a single-device layer, bit for bit (every
    expert row is the same products in the same order, whichever block it sits in)."""
    from expert_routing_router_b300 import moe
    w, R, G, static = OVERLAP_CASES[name]
    ranks, whole = _ranks(w, R, seed=2, groups=G, static=static)
    plans = ep.run_layer_loopback(ranks, overlap=True)
    torch.cuda.synchronize()
    assert plans[0].G == min(G, R)
    hw = host_weights(whole)
    for r, rank in enumerate(ranks):
        assert int(rank.b.workspace[:4].view(torch.int32).item()) == 0
        assert int(rank.local_ws[:4].view(torch.int32).item()) == 0
        n_tok = None if w.tokens <= 1024 and w.hidden <= 1024 else 96
        one = moe.LayerBuffers(w)
        moe.run_layer(one, rank.inp)
        torch.cuda.synchronize()
        # with an INT8 payload the received rows live on the expert's rank, so the step
        # by step check runs on the single-device layer, which this rank must equal
        check_layer(w, rank.inp, one if w.payload == "int8" else rank.b,
                    n_sample_tokens=n_tok,
                    n_sample_rows=None if n_tok is None else "borders", seed=r, hw=hw)
        assert torch.equal(rank.b.out, one.out), f"rank {r}: overlapped layer differs"


def test_static_plan_moves_no_counts_and_repeats_exactly():
    """The fixed plan is built once: two layer steps give identical outputs, and the
    receive layout, split sizes and segment tables do not change between them."""
    w, R, G, static = OVERLAP_CASES["four_ranks_four_groups_static"]
    ranks, _ = _ranks(w, R, seed=5, groups=G, static=static)
    tabs = [(r.g_start.clone(), r.g_kept.clone()) for r in ranks]
    p1 = ep.run_layer_loopback(ranks, overlap=True)
    torch.cuda.synchronize()
    out1 = [r.b.out.clone() for r in ranks]
    p2 = ep.run_layer_loopback(ranks, overlap=True)
    torch.cuda.synchronize()
    for r, rank in enumerate(ranks):
        assert p1[r] is p2[r] is rank.static_plan
        assert torch.equal(rank.g_start, tabs[r][0]) and torch.equal(rank.g_kept, tabs[r][1])
        assert torch.equal(rank.b.out, out1[r])


def test_expert_parallel_layer_dist_single_rank_static_plan():
    """run_layer_dist with the fixed plan (capacity-padded send buffer) through an NCCL
    group of one rank: no count exchange, every chunk a whole expert block."""
    import socket
    import torch.distributed as dist
    w, _, _, _ = OVERLAP_CASES["four_ranks_four_groups_static"]
    w = dataclasses.replace(w, num_ranks=1, rank_map=0)
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                            world_size=1)
    try:
        ranks, whole = _ranks(w, 1, seed=8, groups=2, static=True)
        plan = ep.run_layer_dist(ranks[0])
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    r = ranks[0]
    assert plan is r.static_plan and plan.G == 1
    assert int(r.local_ws[:4].view(torch.int32).item()) == 0
    check_layer(w, r.inp, r.b)
