"""Writes stay inside their rows (a stand-in for a race / out-of-bounds detector, which
is not available on this GPU): every output buffer is filled with a canary bit pattern
before the layer runs, and afterwards
  * every row the layer must produce holds no canary (it was written), and
  * every row that holds no assignment — send-buffer rows past num_kept (packed
    layout), padding rows of the capacity-padded layout, and their INT8 codes and
    scales — still holds the canary (nothing wrote it).
"""
import numpy as np
import pytest
import torch

from expert_routing_router_b300 import workloads as W
from test_gpu_parity import host, small

pytestmark = pytest.mark.gpu

CANARY16 = 0x7FA5            # a bf16 NaN bit pattern no kernel produces
CANARY32 = 0x7FA5A5A5        # the fp32 counterpart


def _fill(t):
    if t is None:
        return
    if t.dtype == torch.bfloat16:
        t.view(torch.int16).fill_(CANARY16)
    elif t.dtype == torch.float32:
        t.view(torch.int32).fill_(CANARY32)
    elif t.dtype == torch.int8:
        t.fill_(-128)              # codes are clamped to +-127, so -128 is never written
    else:
        t.fill_(-7)


def _is_canary(rows):
    a = host(rows)
    if a.dtype == np.uint16:
        return a == CANARY16
    if a.dtype == np.float32:
        return a.view(np.int32) == CANARY32
    if a.dtype == np.int8:
        return a == -128
    return a == -7


CASES = {
    "packed_capacity_drops": small(tokens=700, hidden=136, num_experts=12, top_k=3, num_ranks=3,
                                   score_fn=0, num_groups=1, topk_groups=1, capacity_factor=0.7,
                                   d_ff=96, shared_d_ff=64, sel_bias_std=0.0),
    "capacity_padded": small(tokens=500, hidden=128, num_experts=8, top_k=2, num_ranks=4,
                             score_fn=0, num_groups=1, topk_groups=1, capacity_factor=1.3,
                             d_ff=64, shared_d_ff=0, sel_bias_std=0.0, dispatch_mode=1),
    "decode_sized": small(tokens=9, hidden=264, num_experts=64, top_k=4, num_ranks=8,
                          num_groups=8, topk_groups=4, d_ff=200, shared_d_ff=72),
    "sm_pairs": small(tokens=1500, hidden=264, num_experts=4, top_k=2, num_ranks=2,
                      num_groups=2, topk_groups=1, d_ff=200, shared_d_ff=72,
                      capacity_factor=0.9),
    "int8_payload_drops": small(tokens=600, hidden=264, num_experts=16, top_k=4, num_ranks=4,
                                capacity_factor=0.8, d_ff=200, shared_d_ff=72, payload="int8"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_writes_stay_in_their_rows(name, moe_lib):
    moe = moe_lib
    w = CASES[name]
    inp = W.make_inputs(w, seed=13, device="cuda")
    b = moe.LayerBuffers(w)
    outs = ["xperm", "yperm", "out", "logits", "topk_w", "yshared", "xperm_q", "xscale",
            "yperm_q", "yscale"]
    for n in outs:
        _fill(getattr(b, n))
    moe.run_layer(b, inp)
    torch.cuda.synchronize()
    assert int(b.workspace[:4].view(torch.int32).item()) == 0
    ps = host(b.perm_src)
    held = ps >= 0                         # send-buffer rows that hold an assignment
    assert held.sum() == int(b.num_kept.item())
    # produced in full
    for n in ("out", "logits", "topk_w") + (("yshared",) if w.shared_d_ff else ()):
        assert not _is_canary(getattr(b, n)).any(), n
    # send and return rows: written where an assignment is held, untouched elsewhere
    bufs = ["xperm_q", "xscale", "yperm_q", "yscale"] if b.int8_payload else []
    bufs += ["xperm", "yperm"]
    for n in bufs:
        c = _is_canary(getattr(b, n))
        c = c.reshape(c.shape[0], -1)
        assert not c[held].any(), n
        assert c[~held].all(), f"{n}: a row without an assignment was written"
