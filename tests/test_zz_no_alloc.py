"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc or hand over a workspace (a
runtime whose device memory is planned ahead by an allocator it does not control,
or a path on which an allocation, which may synchronise the device, is not
allowed).  For them moe_dispatch_noalloc keeps its scratch in a static device array
inside the library.  This test calls it through the C ABI twice in a row, on two
different routings, and checks every output against moe_dispatch (bit-exact: all
outputs are integers or copied rows).  It must pass alone in a fresh process and
after the other tests.
"""
import dataclasses

import numpy as np
import pytest
import torch

from expert_routing_router_b300 import workloads as W

pytestmark = pytest.mark.gpu

OUTS = ("xperm", "expert_counts", "kept_counts", "expert_start", "rank_counts", "rank_offsets",
        "slot_of", "perm_src", "num_kept")


def _route(moe, b, inp):
    moe.moe_route(b.cfg, inp["x"], inp["w_router"], inp["b_router"], inp["sel_bias"], b.logits,
                  b.topk_idx, b.topk_w, b.workspace)


def _outputs(moe, w):
    return {n: getattr(moe.LayerBuffers(w), n) for n in OUTS}


def test_dispatch_noalloc_matches_dispatch_twice(moe_lib):
    moe = moe_lib
    w = W.Workload("noalloc", tokens=5000, hidden=200, num_experts=24, top_k=3, num_ranks=5,
                   rank_map=1, score_fn=0, normalize_topk=False, num_groups=1, topk_groups=1,
                   capacity_factor=1.1, d_ff=64, shared_d_ff=0, act_dtype="bf16",
                   router_offset_std=1.0, sel_bias_std=0.0, bias_step=0.0)
    b = moe.LayerBuffers(w)
    for seed in (21, 22):                         # two calls in a row, different routings
        inp = W.make_inputs(w, seed=seed, device="cuda", with_experts=False)
        _route(moe, b, inp)
        ref = _outputs(moe, w)
        moe.moe_dispatch(b.cfg, b.topk_idx, inp["x"], ref["xperm"], ref["expert_counts"],
                         ref["kept_counts"], ref["expert_start"], ref["rank_counts"],
                         ref["rank_offsets"], ref["slot_of"], ref["perm_src"], ref["num_kept"],
                         b.workspace)
        got = _outputs(moe, w)
        for t in got.values():
            t.fill_(-7) if t.dtype == torch.int32 else t.zero_()
        moe.moe_dispatch_noalloc(b.cfg, b.topk_idx, inp["x"], got["xperm"], got["expert_counts"],
                                 got["kept_counts"], got["expert_start"], got["rank_counts"],
                                 got["rank_offsets"], got["slot_of"], got["perm_src"],
                                 got["num_kept"])
        torch.cuda.synchronize()
        nk = int(ref["num_kept"].item())
        assert 0 < nk < w.tokens * w.top_k        # the cap dropped some assignments
        for n in OUTS:
            r, g = ref[n], got[n]
            if n == "xperm":
                r, g = r[:nk], g[:nk]
            assert torch.equal(r, g), n


def test_dispatch_noalloc_at_its_scratch_limit(moe_lib):
    """A layer whose histogram fills the static array exactly: 65,536 tokens at top-8
    over 256 experts is 256 chunks of 2048 assignments x 256 experts = 65,536 int32."""
    moe = moe_lib
    w = W.Workload("noalloc_limit", tokens=65536, hidden=64, num_experts=256, top_k=8,
                   num_ranks=64, rank_map=0, score_fn=1, normalize_topk=True, num_groups=8,
                   topk_groups=4, capacity_factor=0.0, d_ff=64, shared_d_ff=0,
                   act_dtype="bf16", router_offset_std=0.0, sel_bias_std=0.1, bias_step=0.0)
    assert -(-w.tokens * w.top_k // 2048) * w.num_experts == 65536
    b = moe.LayerBuffers(w)
    inp = W.make_inputs(w, seed=23, device="cuda", with_experts=False)
    _route(moe, b, inp)
    ref = _outputs(moe, w)
    moe.moe_dispatch(b.cfg, b.topk_idx, inp["x"], ref["xperm"], ref["expert_counts"],
                     ref["kept_counts"], ref["expert_start"], ref["rank_counts"],
                     ref["rank_offsets"], ref["slot_of"], ref["perm_src"], ref["num_kept"],
                     b.workspace)
    for _ in range(2):
        got = _outputs(moe, w)
        for t in got.values():
            t.fill_(-7) if t.dtype == torch.int32 else t.zero_()
        moe.moe_dispatch_noalloc(b.cfg, b.topk_idx, inp["x"], got["xperm"], got["expert_counts"],
                                 got["kept_counts"], got["expert_start"], got["rank_counts"],
                                 got["rank_offsets"], got["slot_of"], got["perm_src"],
                                 got["num_kept"])
        torch.cuda.synchronize()
        assert int(ref["num_kept"].item()) == w.tokens * w.top_k
        for n in OUTS:
            assert torch.equal(ref[n], got[n]), n
    # one chunk more than the array holds: 257 chunks x 256 experts
    big = moe.config(dataclasses.replace(w, tokens=w.tokens + 1))
    with pytest.raises(moe.MoeError) as e:
        moe.moe_dispatch_noalloc(big, *[torch.empty(4, dtype=torch.int32, device="cuda")] * 11)
    assert e.value.status == moe.MOE_ERR_WORKSPACE


def test_dispatch_noalloc_rejects_layers_beyond_its_scratch(moe_lib):
    cfg = moe_lib.config(W.DSV3_PREFILL.with_tokens(70000))   # 274 chunks x 256 experts
    with pytest.raises(moe_lib.MoeError) as e:
        moe_lib.moe_dispatch_noalloc(cfg, *[torch.empty(4, dtype=torch.int32, device="cuda")] * 11)
    assert e.value.status == moe_lib.MOE_ERR_WORKSPACE
