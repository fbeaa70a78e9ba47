"""The C-ABI library loads without a GPU, exports every declared entry point, and
rejects bad arguments on the host before anything touches a device (CPU only)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from expert_routing_router_b300 import workloads as W


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(moe_lib):
    names = _declared()
    assert {"moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_bias_update",
            "moe_workspace_size", "moe_status_string"} <= names
    raw = ctypes.CDLL(moe_lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings(moe_lib):
    for s in range(5):
        assert moe_lib.status_string(s).startswith("MOE_")
    assert "unknown" in moe_lib.status_string(99)


def test_workspace_size_grows_with_layer(moe_lib):
    a = moe_lib.moe_workspace_size(moe_lib.config(W.SWITCH_TOP1))
    b = moe_lib.moe_workspace_size(moe_lib.config(W.DSV3_PREFILL))
    assert 0 < a < b
    # the FFN intermediate dominates: (N*k*F + N*Fs) bf16 for the DeepSeek-V3 prefill layer
    assert b >= (8192 * 8 * 2048 + 8192 * 2048) * 2


FAKE = 1 << 20  # an aligned, never-dereferenced address: validation fails before any use


def _route(moe, cfg, ws_bytes=1 << 40, x=FAKE, ws=FAKE, wr=FAKE):
    P = ctypes.c_void_p
    return moe.lib.moe_route(ctypes.byref(cfg), P(x), P(wr), None, None, P(FAKE), P(FAKE),
                             P(FAKE), P(ws), ws_bytes, None)


@pytest.mark.parametrize("field,value", [
    ("tokens", 0), ("hidden", 12), ("hidden", 4), ("num_experts", 257), ("num_experts", 0),
    ("top_k", 0), ("top_k", 9), ("num_ranks", 0), ("num_ranks", 300), ("rank_map", 2),
    ("score_fn", 3), ("num_groups", 3), ("topk_groups", 9), ("d_ff", 12), ("shared_d_ff", 4),
    ("act_dtype", 5), ("capacity_factor", float("inf")), ("dispatch_mode", 2),
    # 256 experts: more weight rows than 32-bit coordinates reach
    ("d_ff", 1 << 23), ("hidden", 1 << 23), ("shared_d_ff", 1 << 30)])
def test_invalid_config_rejected_on_host(moe_lib, field, value):
    cfg = moe_lib.config(W.DSV3_PREFILL)
    setattr(cfg, field, value)
    assert _route(moe_lib, cfg) == moe_lib.MOE_ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    assert moe_lib.lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == \
        moe_lib.MOE_ERR_INVALID_ARG


def test_padded_dispatch_needs_capacity_and_sizes_send_rows(moe_lib):
    cfg = moe_lib.config(W.GSHARD_TOP2_PADDED)
    assert moe_lib.moe_send_rows(cfg) == 64 * 1280          # E * C
    assert moe_lib.moe_send_rows(moe_lib.config(W.GSHARD_TOP2)) == 32768 * 2
    cfg.capacity_factor = 0.0                               # no capacity, no padded layout
    assert _route(moe_lib, cfg) == moe_lib.MOE_ERR_INVALID_ARG


def test_group_limit_must_leave_k_candidates(moe_lib):
    cfg = moe_lib.config(W.DSV3_PREFILL)
    cfg.topk_groups = 1          # 1 group of 32 experts still leaves 8 candidates: fine
    cfg.num_groups = 64          # 1 group of 4 experts < top-8: rejected
    assert _route(moe_lib, cfg) == moe_lib.MOE_ERR_INVALID_ARG


def test_contiguous_rank_map_needs_divisor(moe_lib):
    cfg = moe_lib.config(W.DSV3_PREFILL)
    cfg.num_ranks = 40           # 256 % 40 != 0: only the round-robin map accepts it
    assert _route(moe_lib, cfg) == moe_lib.MOE_ERR_INVALID_ARG


def test_null_misaligned_and_small_workspace(moe_lib):
    cfg = moe_lib.config(W.SWITCH_TOP1)
    assert _route(moe_lib, cfg, x=0) == moe_lib.MOE_ERR_INVALID_ARG
    assert _route(moe_lib, cfg, x=FAKE + 8) == moe_lib.MOE_ERR_INVALID_ARG   # not 16-byte aligned
    assert _route(moe_lib, cfg, ws=FAKE + 16) == moe_lib.MOE_ERR_INVALID_ARG  # not 256-byte aligned
    need = moe_lib.moe_workspace_size(cfg)
    assert _route(moe_lib, cfg, ws_bytes=need - 1) == moe_lib.MOE_ERR_WORKSPACE
    P = ctypes.c_void_p
    # dispatch without a send buffer is allowed; with one, x must be given
    rc = moe_lib.lib.moe_dispatch(ctypes.byref(cfg), P(FAKE), None, P(FAKE), *[P(FAKE)] * 8,
                                  P(FAKE), need, None)
    assert rc == moe_lib.MOE_ERR_INVALID_ARG
    # expert FFN of a layer with a shared expert needs the shared weights
    c3 = moe_lib.config(W.DSV3_PREFILL)
    rc = moe_lib.lib.moe_expert_ffn(ctypes.byref(c3), *[P(FAKE)] * 5, P(FAKE), None, None,
                                    P(FAKE), P(FAKE), P(FAKE),
                                    moe_lib.moe_workspace_size(c3), None)
    assert rc == moe_lib.MOE_ERR_INVALID_ARG
    assert moe_lib.lib.moe_bias_update(ctypes.byref(cfg), None, P(FAKE), ctypes.c_float(1e-3),
                                       None) == moe_lib.MOE_ERR_INVALID_ARG
    assert moe_lib.lib.moe_bias_update(ctypes.byref(cfg), P(FAKE), P(FAKE),
                                       ctypes.c_float(float("nan")), None) == \
        moe_lib.MOE_ERR_INVALID_ARG
    assert moe_lib.lib.moe_combine(None, P(FAKE), P(FAKE), P(FAKE), None, None, P(FAKE),
                                   None) == moe_lib.MOE_ERR_INVALID_ARG


def test_int8_payload_calls_validate_on_host(moe_lib):
    """The INT8 payload calls reject null and misaligned buffers before any launch."""
    P = ctypes.c_void_p
    cfg = moe_lib.config(W.DSV3_PREFILL_INT8)
    need = moe_lib.moe_workspace_size(cfg)
    L = moe_lib.lib
    # dispatch_q8: missing codes buffer, misaligned codes buffer, small workspace
    assert L.moe_dispatch_q8(ctypes.byref(cfg), P(FAKE), P(FAKE), None, P(FAKE),
                             *[P(FAKE)] * 8, P(FAKE), need, None) == moe_lib.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch_q8(ctypes.byref(cfg), P(FAKE), P(FAKE), P(FAKE + 8), P(FAKE),
                             *[P(FAKE)] * 8, P(FAKE), need, None) == moe_lib.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch_q8(ctypes.byref(cfg), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                             *[P(FAKE)] * 8, P(FAKE), need - 1, None) == moe_lib.MOE_ERR_WORKSPACE
    # quant / dequant: null perm_src, misaligned rows, misaligned scale
    assert L.moe_quant_rows(ctypes.byref(cfg), P(FAKE), None, P(FAKE), P(FAKE),
                            None) == moe_lib.MOE_ERR_INVALID_ARG
    assert L.moe_quant_rows(ctypes.byref(cfg), P(FAKE + 8), P(FAKE), P(FAKE), P(FAKE),
                            None) == moe_lib.MOE_ERR_INVALID_ARG
    assert L.moe_dequant_rows(ctypes.byref(cfg), P(FAKE), P(FAKE + 2), P(FAKE), P(FAKE),
                              None) == moe_lib.MOE_ERR_INVALID_ARG
    assert L.moe_dequant_rows(None, P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                              None) == moe_lib.MOE_ERR_INVALID_ARG
    # combine_q8: missing scales, misaligned residual
    assert L.moe_combine_q8(ctypes.byref(cfg), P(FAKE), None, P(FAKE), P(FAKE), P(FAKE), None,
                            P(FAKE), None) == moe_lib.MOE_ERR_INVALID_ARG
    assert L.moe_combine_q8(ctypes.byref(cfg), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE + 4),
                            None, P(FAKE), None) == moe_lib.MOE_ERR_INVALID_ARG


def test_backward_calls_validate_on_host(moe_lib):
    """Backward entry points: fp32 expert backward is unsupported, bad buffers are
    rejected, and the workspace size covers the recomputed activations."""
    P = ctypes.c_void_p
    L = moe_lib.lib
    c3 = moe_lib.config(W.DSV3_PREFILL)
    need = moe_lib.moe_backward_workspace_size(c3)
    # g, u, h and [dg | du] in bf16 for the send rows and the shared expert's tokens
    assert need >= 2 * 5 * (8192 * 8 * 2048 + 8192 * 2048)
    c0 = moe_lib.config(W.TINY_TOP2_F32)
    n0 = moe_lib.moe_backward_workspace_size(c0)
    args = [P(FAKE)] * 16 + [None]      # every pointer before the workspace; no saved
    assert L.moe_expert_ffn_backward(ctypes.byref(c0), *args, P(FAKE), n0, None) == \
        moe_lib.MOE_ERR_UNSUPPORTED
    assert L.moe_expert_ffn_backward(ctypes.byref(c3), *args, P(FAKE), need - 1, None) == \
        moe_lib.MOE_ERR_WORKSPACE
    bad = list(args)
    bad[9] = None                       # the shared expert's dout is required
    assert L.moe_expert_ffn_backward(ctypes.byref(c3), *bad, P(FAKE), need, None) == \
        moe_lib.MOE_ERR_INVALID_ARG
    assert L.moe_combine_backward(ctypes.byref(c3), P(FAKE + 8), *[P(FAKE)] * 5, None) == \
        moe_lib.MOE_ERR_INVALID_ARG
    # router: dW and db come as a pair
    assert L.moe_route_backward(ctypes.byref(c3), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                P(FAKE), None, P(FAKE), None, P(FAKE), need,
                                None) == moe_lib.MOE_ERR_INVALID_ARG
    # router weight gradient: the backward workspace is required and checked for size
    assert L.moe_route_backward(ctypes.byref(c3), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                P(FAKE), None, P(FAKE), P(FAKE), None, 0,
                                None) == moe_lib.MOE_ERR_INVALID_ARG
    assert L.moe_route_backward(ctypes.byref(c3), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                P(FAKE), None, P(FAKE), P(FAKE), P(FAKE), need - 1,
                                None) == moe_lib.MOE_ERR_WORKSPACE
    assert L.moe_dispatch_backward(ctypes.byref(c3), P(FAKE), P(FAKE), None, None, None, P(FAKE),
                                   None) == moe_lib.MOE_ERR_INVALID_ARG
