"""Device-side failure handling, tested without faulting or hanging the GPU.

Every mbarrier wait in the tensor-core kernels has a limit of about 2 s.  The
self-test entry point makes one wait run out on purpose (one pipeline slot is armed
but never loaded); the kernel must report it through the workspace status word,
finish in bounded time, and leave the CUDA context usable for a normal layer call.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from expert_routing_router_b300 import workloads as W

pytestmark = pytest.mark.gpu


def _host(t):
    t = t.detach().contiguous().cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def test_stalled_pipeline_reports_status_and_context_survives(moe_lib):
    moe = moe_lib
    w = W.Workload("stall", tokens=1000, hidden=256, num_experts=16, top_k=4, num_ranks=4,
                   rank_map=0, score_fn=0, normalize_topk=True, num_groups=1, topk_groups=1,
                   capacity_factor=0.0, d_ff=128, shared_d_ff=0, act_dtype="bf16",
                   router_offset_std=0.0, sel_bias_std=0.0, bias_step=0.0, expert_std=0.05)
    inp = W.make_inputs(w, seed=9, device="cuda")
    b = moe.LayerBuffers(w)
    c = b.cfg
    moe.moe_route(c, inp["x"], inp["w_router"], inp["b_router"], None, b.logits, b.topk_idx,
                  b.topk_w, b.workspace)
    moe.moe_dispatch(c, b.topk_idx, inp["x"], b.xperm, b.expert_counts, b.kept_counts,
                     b.expert_start, b.rank_counts, b.rank_offsets, b.slot_of, b.perm_src,
                     b.num_kept, b.workspace)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.moe_selftest_ffn_stall(c, b.xperm, b.expert_start, b.kept_counts, inp["w_gate_up"],
                               inp["w_down"], None, None, None, b.yperm, None, b.workspace)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    status = int(b.workspace[:4].view(torch.int32).item())
    assert status == 3, status          # the MMA issuer's wait for the never-loaded slot
    assert 1.5 < dt < 20.0, dt          # gave up after its ~2 s limit, did not hang

    # the context is still usable: a normal layer on the same buffers is correct
    b.workspace[:256].zero_()
    moe.run_layer(b, inp)
    torch.cuda.synchronize()
    assert int(b.workspace[:4].view(torch.int32).item()) == 0
    idx = _host(b.topk_idx)
    wts = _host(b.topk_w).astype(np.float64)
    d = oracle.dispatch(idx, w.num_experts, w.num_ranks, w.rank_map, 0.0)
    toks = np.arange(0, w.tokens, 7, dtype=np.int32)
    ref = oracle.layer_tokens(toks, _host(inp["x"]), idx, wts, d["slot_of"],
                              _host(inp["w_gate_up"]), _host(inp["w_down"]))
    got = b.out.double().cpu().numpy()[toks]
    assert np.abs(got - ref).max() <= 2e-2 * np.abs(ref).max()
