"""GPU parity: every step of the CUDA path against the CPU oracle (needs a B300).

Per step, the oracle gets the very inputs the GPU step got, so each comparison
isolates one kernel:
  logits            oracle fp64 logits of the same x, W, b          max-abs rel 1e-5
  routing           oracle routing of the GPU's own logits          bit-exact indices,
                                                                    weights rel 1e-5
  dispatch tables   oracle dispatch of the GPU's own top-k ids      bit-exact
  send buffer       xperm[s] == x[perm_src[s] // k]                 bit-exact
  expert FFN        oracle fp64 FFN of the GPU's xperm rows         1e-4 (fp32) / 2e-2 (bf16)
  combine           oracle fp64 sum of the GPU's yperm / weights    one output rounding
  layer             oracle fp64 layer from x and the weights        1e-4 (fp32) / 2e-2 (bf16)
  bias update       oracle fp32 sign rule                           bit-exact
Tolerances are max-abs normalised: max|got - ref| <= tol * max|ref|.  Full-size
workloads are checked on every expert's first and last send row and the rows on both
sides of every 128-row tile border (the same for the shared expert's token rows), and
the whole layer on a seeded sample of at least 1,024 tokens that always includes every
token whose choices were all dropped; the small cases and the decode batches are
checked in full.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from expert_routing_router_b300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_LOGITS = 1e-5
TOL_W = 1e-5
TOL_OUT = {"f32": 1e-4, "bf16": 2e-2}
TOL_COMBINE = {"f32": 2e-6, "bf16": 4e-3}


def host(t):
    """Tensor -> numpy: fp32 as float32, bf16 as uint16 bit patterns."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def f64(t):
    return t.detach().cpu().double().numpy()


def close(got, ref, tol, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.max(np.abs(got - ref)) if got.size else 0.0
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    assert err <= tol * scale, f"{what}: max|err| {err:.3e} > {tol} * max|ref| {scale:.3e}"
    return err / scale if scale else 0.0


def run_gpu(w, inp):
    from expert_routing_router_b300 import moe
    b = moe.LayerBuffers(w)
    bias_before = None if inp["sel_bias"] is None else inp["sel_bias"].clone()
    moe.run_layer(b, inp)
    torch.cuda.synchronize()
    # device status word (first int32 of the workspace): no kernel gave up a wait
    assert int(b.workspace[:4].view(torch.int32).item()) == 0
    return b, bias_before


def host_weights(inp):
    """Host copies of the expert weights (made once per input set)."""
    return {k: None if inp[k] is None else host(inp[k])
            for k in ("w_gate_up", "w_down", "shared_gate_up", "shared_down")}


def check_route_dispatch(w, inp, b, rng, n_sample_tokens):
    """Logits, routing and dispatch tables (shared by both payload paths)."""
    N, k, E = w.tokens, w.top_k, w.num_experts
    x_h = host(inp["x"])
    # ---- logits (sampled rows at full size)
    rows = np.arange(N) if n_sample_tokens is None else np.sort(
        rng.choice(N, size=min(N, 4 * n_sample_tokens), replace=False))
    ref_l = oracle.router_logits(x_h[rows], host(inp["w_router"]), host(inp["b_router"]))
    got_l = host(b.logits)
    close(got_l[rows], ref_l, TOL_LOGITS, "router logits")
    # ---- routing from the GPU's own logits: bit-exact ids
    sb = None if inp["sel_bias"] is None else host(inp["sel_bias"])
    idx_ref, w_ref = oracle.route(got_l, k, w.score_fn, w.normalize_topk, w.num_groups,
                                  w.topk_groups, sb)
    idx_gpu = host(b.topk_idx)
    mism = np.argwhere(idx_gpu != idx_ref)
    assert mism.size == 0, f"top-k ids differ at {mism[:5].tolist()}"
    close(host(b.topk_w), w_ref, TOL_W, "combine weights")
    # ---- dispatch tables from the GPU's own ids: bit-exact
    d = oracle.dispatch(idx_gpu, E, w.num_ranks, w.rank_map, w.capacity_factor,
                        mode=w.dispatch_mode)
    for name in ("expert_counts", "kept_counts", "expert_start", "rank_counts", "rank_offsets",
                 "slot_of", "perm_src"):
        np.testing.assert_array_equal(host(getattr(b, name)), d[name], err_msg=name)
    nk = int(host(b.num_kept)[0])
    assert nk == d["num_kept"]
    assert host(b.expert_counts).sum() == N * k
    kept_rows = np.nonzero(d["perm_src"] >= 0)[0]
    assert kept_rows.size == nk
    return x_h, idx_gpu, w_ref, d, nk, kept_rows


def sample_tokens(rng, N, n_sample_tokens, d, k, max_dropped=32):
    """Token sample (or all), always including fully dropped tokens (up to max_dropped)."""
    slot = d["slot_of"].reshape(N, k)
    dropped = np.nonzero((slot < 0).all(axis=1))[0]
    if n_sample_tokens is None:
        toks = np.arange(N)
    else:
        toks = np.unique(np.concatenate([rng.choice(N, size=min(N, n_sample_tokens), replace=False),
                                         dropped[:max_dropped]]))
    return toks.astype(np.int32), dropped


TILE = 128  # row tile of the single-SM expert kernels; the SM-pair tiles (256) are multiples


def border_rows(start, count, tile=TILE):
    """Rows start..start+count-1 that a tiled kernel handles at an edge: the first and
    last row, and the rows on both sides of every tile border inside the segment."""
    if count <= 0:
        return np.zeros(0, np.int64)
    local = {0, count - 1}
    for b in range(tile, count, tile):
        local.update((b - 1, b))
    return start + np.array(sorted(local), np.int64)


def stratified_rows(expert_start, kept_counts):
    """Send rows at the edges of every expert segment and of its row tiles."""
    parts = [border_rows(int(s), int(c)) for s, c in zip(expert_start, kept_counts)]
    return np.unique(np.concatenate(parts)) if parts else np.zeros(0, np.int64)


# relative rounding of one store to the output type (round to nearest: half an ulp,
# taken as a full ulp to cover the last fp32 additions before the store)
OUT_ROUNDING = {"f32": 2.0 ** -23, "bf16": 2.0 ** -8}


def check_layer_output(w, out_got, x_h, toks, l_ref):
    """The layer output, and the MoE delta (out - x), against the oracle's layer.  The
    delta gate keeps an FFN error from hiding behind the residual: elementwise
    |got - ref| <= tol * max|delta_ref| + (output rounding) * |out_ref|, the second
    term being the storage rounding of out itself, which a small delta cannot absorb."""
    rel = close(out_got[toks], l_ref, TOL_OUT[w.act_dtype], "layer output")
    xt = x_h[toks].astype(np.float64) if w.act_dtype == "f32" else bf16_to_f64(x_h[toks])
    d_got, d_ref = out_got[toks] - xt, l_ref - xt
    if d_ref.size:
        allow = TOL_OUT[w.act_dtype] * np.max(np.abs(d_ref)) + \
            OUT_ROUNDING[w.act_dtype] * np.abs(l_ref)
        bad = np.abs(d_got - d_ref) > allow
        assert not bad.any(), (f"layer delta (out - x): {int(bad.sum())} elements off, worst "
                               f"{np.max(np.abs(d_got - d_ref) - allow):.3e} beyond the allowance; "
                               f"max|delta_ref| {np.max(np.abs(d_ref)):.3e}")
    return rel


def bf16_to_f64(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_layer(w, inp, b, n_sample_tokens=None, n_sample_rows=None, seed=0, hw=None):
    """All per-step and end-to-end checks for one layer call."""
    if getattr(w, "payload", "act") == "int8":
        return check_layer_int8(w, inp, b, n_sample_tokens, n_sample_rows, seed, hw)
    if hw is None:
        hw = host_weights(inp)
    rng = np.random.default_rng(seed)
    N, k, E = w.tokens, w.top_k, w.num_experts
    x_h, idx_gpu, w_ref, d, nk, kept_rows = check_route_dispatch(w, inp, b, rng, n_sample_tokens)
    # ---- send buffer rows are exact copies (the rows that hold an assignment)
    ps = d["perm_src"][kept_rows]
    xp = host(b.xperm[torch.from_numpy(kept_rows).cuda().long()]) if nk else x_h[:0]
    np.testing.assert_array_equal(xp, x_h[ps // k], err_msg="xperm")
    # ---- expert FFN on the GPU's send rows
    flat_idx = idx_gpu.reshape(-1)
    if n_sample_rows == "borders":
        # every expert segment's edges and row-tile borders, as positions in kept_rows
        srows = stratified_rows(d["expert_start"], d["kept_counts"])
        sel = np.searchsorted(kept_rows, srows)
        assert np.array_equal(kept_rows[sel], srows)
    else:
        sel = np.arange(nk) if n_sample_rows is None else np.sort(
            rng.choice(nk, size=min(nk, n_sample_rows), replace=False))
    wgu, wd, sgu, sd = hw["w_gate_up"], hw["w_down"], hw["shared_gate_up"], hw["shared_down"]
    if sel.size:
        y_ref = oracle.expert_rows(xp[sel], flat_idx[ps[sel]], wgu, wd)
        y_got = f64(b.yperm[torch.from_numpy(kept_rows[sel]).cuda().long()])
        close(y_got, y_ref, TOL_OUT[w.act_dtype], "expert FFN rows")
    if sgu is not None:
        if n_sample_rows == "borders":
            trows = border_rows(0, N)
        else:
            trows = np.arange(N) if n_sample_rows is None else np.sort(
                rng.choice(N, size=min(N, n_sample_rows), replace=False))
        ys_ref = oracle.expert_rows(x_h[trows], np.full(trows.size, E, np.int32), wgu, wd, sgu, sd)
        close(f64(b.yshared[torch.from_numpy(trows).cuda().long()]), ys_ref, TOL_OUT[w.act_dtype],
              "shared expert rows")
    # ---- combine from the GPU's yperm / weights, and the whole layer
    toks, dropped = sample_tokens(rng, N, n_sample_tokens, d, k,
                                  max_dropped=N if n_sample_tokens is not None else 32)
    ys_h = None if b.yshared is None else host(b.yshared)
    out_got = f64(b.out)
    c_ref = oracle.combine(toks, x_h, host(b.yperm), d["slot_of"],
                           host(b.topk_w).astype(np.float64), ys_h)
    close(out_got[toks], c_ref, TOL_COMBINE[w.act_dtype], "combine")
    if w.shared_d_ff == 0 and dropped.size:
        # a token whose every choice was dropped leaves the layer unchanged, bit for bit
        np.testing.assert_array_equal(host(b.out)[dropped], x_h[dropped])
    l_ref = oracle.layer_tokens(toks, x_h, idx_gpu, w_ref, d["slot_of"], wgu, wd, sgu, sd)
    rel = check_layer_output(w, out_got, x_h, toks, l_ref)
    return dict(rel_err=rel, drop_rate=1.0 - nk / (N * k), num_kept=nk)


def check_layer_int8(w, inp, b, n_sample_tokens=None, n_sample_rows=None, seed=0, hw=None):
    """The INT8-payload path, step by step:
      send codes/scales   oracle quantisation of the kept tokens' rows     bit-exact
      received rows       oracle dequantisation of the GPU's codes         bit-exact
      expert FFN          oracle fp64 FFN of the GPU's received rows       as check_layer
      return codes/scales oracle quantisation of the GPU's expert rows     bit-exact
      combine             oracle fp64 sum of the GPU's return payload      one output rounding
      layer               oracle layer with the routed experts fed the dequantised rows,
                          expert outputs unquantised; the allowance adds one code step
                          of the return payload per kept choice."""
    if hw is None:
        hw = host_weights(inp)
    rng = np.random.default_rng(seed)
    N, k, E = w.tokens, w.top_k, w.num_experts
    x_h, idx_gpu, w_ref, d, nk, kept_rows = check_route_dispatch(w, inp, b, rng, n_sample_tokens)
    ps = d["perm_src"][kept_rows]
    if n_sample_rows == "borders":
        srows = stratified_rows(d["expert_start"], d["kept_counts"])
        sel = np.searchsorted(kept_rows, srows)
        assert np.array_equal(kept_rows[sel], srows)
    else:
        sel = np.arange(nk) if n_sample_rows is None else np.sort(
            rng.choice(nk, size=min(nk, n_sample_rows), replace=False))
    rows = kept_rows[sel]
    rows_t = torch.from_numpy(rows).cuda().long()
    # ---- send payload: codes and scales of the kept tokens' rows
    q_ref, s_ref = oracle.quant_rows(x_h[ps[sel] // k])
    xq = b.xperm_q[rows_t].cpu().numpy()
    np.testing.assert_array_equal(xq, q_ref, err_msg="send codes")
    np.testing.assert_array_equal(b.xscale[rows_t].cpu().numpy(), s_ref, err_msg="send scales")
    # ---- receiver: dequantised rows
    xdq = host(b.xperm[rows_t])
    np.testing.assert_array_equal(xdq, oracle.dequant_rows(xq, s_ref, w.act_dtype),
                                  err_msg="received rows")
    # ---- expert FFN on the received rows
    flat_idx = idx_gpu.reshape(-1)
    wgu, wd, sgu, sd = hw["w_gate_up"], hw["w_down"], hw["shared_gate_up"], hw["shared_down"]
    if sel.size:
        y_ref = oracle.expert_rows(xdq, flat_idx[ps[sel]], wgu, wd)
        close(f64(b.yperm[rows_t]), y_ref, TOL_OUT[w.act_dtype], "expert FFN rows")
        # ---- return payload: codes and scales of the GPU's expert rows
        yq_ref, ys_ref = oracle.quant_rows(host(b.yperm[rows_t]))
        np.testing.assert_array_equal(b.yperm_q[rows_t].cpu().numpy(), yq_ref,
                                      err_msg="return codes")
        np.testing.assert_array_equal(b.yscale[rows_t].cpu().numpy(), ys_ref,
                                      err_msg="return scales")
    # ---- combine from the GPU's return payload
    toks, dropped = sample_tokens(rng, N, n_sample_tokens, d, k,
                                  max_dropped=N if n_sample_tokens is not None else 32)
    ys_h = None if b.yshared is None else host(b.yshared)
    out_got = f64(b.out)
    c_ref = oracle.combine_q8(toks, x_h, b.yperm_q.cpu().numpy(), b.yscale.cpu().numpy(),
                              d["slot_of"], host(b.topk_w).astype(np.float64), ys_h)
    close(out_got[toks], c_ref, TOL_COMBINE[w.act_dtype], "combine (INT8 payload)")
    if w.shared_d_ff == 0 and dropped.size:
        np.testing.assert_array_equal(host(b.out)[dropped], x_h[dropped])
    # ---- layer: routed experts see the dequantised token rows; shared expert and
    # residual see x itself (they never cross the all-to-all)
    q_all, s_all = oracle.quant_rows(x_h[toks])
    xdq_t = oracle.dequant_rows(q_all, s_all, w.act_dtype)
    xdq_full = np.array(x_h, copy=True)
    xdq_full[toks] = xdq_t
    routed = oracle.layer_tokens(toks, xdq_full, idx_gpu, w_ref, d["slot_of"], wgu, wd)
    xdq64 = xdq_t.astype(np.float64) if w.act_dtype == "f32" else bf16_to_f64(xdq_t)
    xt64 = x_h[toks].astype(np.float64) if w.act_dtype == "f32" else bf16_to_f64(x_h[toks])
    l_ref = xt64 + (routed - xdq64)
    if sgu is not None:
        l_ref += oracle.expert_rows(x_h[toks], np.full(toks.size, E, np.int32), wgu, wd, sgu, sd)
    # The reference keeps the expert outputs unquantised.  The return trip moves each
    # kept term by at most one code step of its row (half a step of rounding; one more
    # where the GPU's and the oracle's y straddle a code boundary), so the allowance
    # adds sum_j w_j * s_j per token (s_j: that row's scale) to the usual terms.
    slot = d["slot_of"].reshape(N, k)[toks]
    ysc = b.yscale.cpu().numpy()
    wts = host(b.topk_w).astype(np.float64)[toks]
    qstep = np.where(slot >= 0, wts * ysc[np.maximum(slot, 0)].astype(np.float64), 0.0).sum(1)
    tol = TOL_OUT[w.act_dtype]
    for what, got_v, ref_v in (("layer output", out_got[toks], l_ref),
                               ("layer delta (out - x)", out_got[toks] - xt64, l_ref - xt64)):
        allow = tol * np.max(np.abs(ref_v)) + qstep[:, None] + \
            OUT_ROUNDING[w.act_dtype] * np.abs(l_ref)
        bad = np.abs(got_v - ref_v) > allow
        assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond the allowance"
    rel = np.max(np.abs(out_got[toks] - l_ref)) / max(np.max(np.abs(l_ref)), 1e-300)
    return dict(rel_err=rel, drop_rate=1.0 - nk / (N * k), num_kept=nk)


# ---------------------------------------------------------------- full-size workloads

@pytest.fixture(scope="module")
def dsv3_inputs():
    inp = W.make_inputs(W.DSV3_PREFILL, seed=0, device="cuda")
    yield inp, host_weights(inp)
    del inp
    torch.cuda.empty_cache()


def test_tiny_top2_f32_full():
    w = W.TINY_TOP2_F32
    inp = W.make_inputs(w, seed=0, device="cuda")
    b, _ = run_gpu(w, inp)
    check_layer(w, inp, b)
    # the glossary page's printed ranges hold on the GPU's routing too
    ec, rc = host(b.expert_counts), host(b.rank_counts)
    assert (ec.min(), ec.max(), rc.min(), rc.max()) == (948, 1087, 1968, 2139)


@pytest.mark.parametrize("w", [W.SWITCH_TOP1, W.GSHARD_TOP2, W.GSHARD_TOP2_PADDED],
                         ids=lambda w: w.name)
def test_capacity_workloads(w):
    inp = W.make_inputs(w, seed=0, device="cuda")
    b, _ = run_gpu(w, inp)
    r = check_layer(w, inp, b, n_sample_tokens=1024, n_sample_rows="borders")
    C = oracle.capacity(w.tokens, w.top_k, w.num_experts, w.capacity_factor)
    assert host(b.kept_counts).max() <= C
    print(f"{w.name}: drop rate {r['drop_rate']:.4f}, layer rel err {r['rel_err']:.2e}")


def test_dsv3_prefill_and_bias_update(dsv3_inputs):
    from expert_routing_router_b300 import moe
    w, (inp, hw) = W.DSV3_PREFILL, dsv3_inputs
    b, bias0 = run_gpu(w, inp)
    check_layer(w, inp, b, n_sample_tokens=1024, n_sample_rows="borders", hw=hw)
    counts = host(b.expert_counts)
    moe.moe_bias_update(b.cfg, b.expert_counts, inp["sel_bias"], w.bias_step)
    torch.cuda.synchronize()
    ref = oracle.bias_update(counts, host(bias0), w.tokens, w.top_k, w.bias_step)
    np.testing.assert_array_equal(host(inp["sel_bias"]), ref)
    inp["sel_bias"].copy_(bias0)


def test_dsv3_prefill_graph_replay_matches_direct_calls(dsv3_inputs):
    """Full-size layer in the launch form the benchmark times (CUDA graph replay):
    bit-identical to direct C-ABI calls."""
    from expert_routing_router_b300 import moe
    w, (inp, _) = W.DSV3_PREFILL, dsv3_inputs
    bias0 = inp["sel_bias"].clone()
    b = moe.LayerBuffers(w)
    moe.run_layer(b, inp, bias_step=w.bias_step)
    torch.cuda.synchronize()
    ref_out, ref_bias = b.out.clone(), inp["sel_bias"].clone()
    inp["sel_bias"].copy_(bias0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.run_layer(b, inp, bias_step=w.bias_step)
    inp["sel_bias"].copy_(bias0)
    b.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(b.out, ref_out)
    assert torch.equal(inp["sel_bias"], ref_bias)
    assert int(b.workspace[:4].view(torch.int32).item()) == 0
    inp["sel_bias"].copy_(bias0)
    del b, g
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", W.DECODE_TOKENS)
def test_dsv3_decode_sweep(dsv3_inputs, T):
    w = W.DSV3_DECODE.with_tokens(T)
    inp = dict(dsv3_inputs[0])
    inp["x"] = W.make_tokens(w, T, seed=1, device="cuda")
    b, _ = run_gpu(w, inp)
    # every token and every expert row up to 128 tokens; at 512 every token and the
    # rows at each segment's edges and tile borders
    check_layer(w, inp, b, n_sample_tokens=None, n_sample_rows=None if T <= 128 else "borders",
                hw=dsv3_inputs[1])


# ---------------------------------------------------------------- edge cases (small, full check)

def small(**kw):
    base = dict(name="edge", tokens=1000, hidden=264, num_experts=16, top_k=4, num_ranks=4,
                rank_map=0, score_fn=1, normalize_topk=True, num_groups=4, topk_groups=2,
                capacity_factor=0.0, d_ff=200, shared_d_ff=72, act_dtype="bf16",
                router_offset_std=0.0, sel_bias_std=0.1, bias_step=1e-3, expert_std=0.05)
    base.update(kw)
    return W.Workload(**base)


EDGE = {
    "ragged_sigmoid_groups_shared": small(),
    "ragged_f32_softmax_cap": small(tokens=777, hidden=136, num_experts=12, top_k=3, num_ranks=3,
                                    score_fn=0, num_groups=1, topk_groups=1,
                                    capacity_factor=1.0, d_ff=40, shared_d_ff=0,
                                    act_dtype="f32", sel_bias_std=0.0),
    "one_token": small(tokens=1, hidden=128, num_experts=64, top_k=8, num_ranks=8,
                       num_groups=8, topk_groups=4, d_ff=64, shared_d_ff=64),
    "dense_single_expert": small(tokens=300, hidden=64, num_experts=1, top_k=1, num_ranks=1,
                                 score_fn=0, num_groups=1, topk_groups=1, d_ff=64,
                                 shared_d_ff=0, sel_bias_std=0.0),
    "k_equals_E": small(tokens=200, hidden=64, num_experts=4, top_k=4, num_ranks=2, score_fn=0,
                        num_groups=1, topk_groups=1, d_ff=32, shared_d_ff=0, sel_bias_std=0.0),
    "round_robin_uneven_ranks": small(tokens=513, hidden=96, num_experts=64, top_k=6,
                                      num_ranks=40, rank_map=1, num_groups=1, topk_groups=1,
                                      d_ff=48, shared_d_ff=0),
    "tiny_capacity_most_dropped": small(tokens=640, hidden=64, num_experts=8, top_k=2,
                                        num_ranks=2, score_fn=0, num_groups=1, topk_groups=1,
                                        capacity_factor=0.05, d_ff=32, shared_d_ff=0,
                                        sel_bias_std=0.0),
    # few rows per expert: the token-major small-segment expert kernel, ragged sizes
    "small_segments_ragged": small(tokens=40, hidden=264, num_experts=64, top_k=4, num_ranks=8,
                                   num_groups=8, topk_groups=4, capacity_factor=1.0, d_ff=200,
                                   shared_d_ff=72),
    # the same kernel with skewed routing: two experts with more than one 32-row token
    # tile (81 rows on the busiest), and a 200-row shared expert (7 token tiles)
    "small_segments_skewed_row_tiles": small(tokens=200, hidden=264, num_experts=64, top_k=1,
                                             num_ranks=8, score_fn=0, num_groups=1,
                                             topk_groups=1, router_offset_std=1.0, d_ff=200,
                                             shared_d_ff=72, sel_bias_std=0.0),
    # decode-sized batches on the token-major kernels: no shared expert; and the
    # capacity-padded layout (each expert's block of C rows at a fixed offset)
    "small_segments_no_shared": small(tokens=3, hidden=264, num_experts=64, top_k=4,
                                      num_ranks=8, num_groups=8, topk_groups=4, d_ff=200,
                                      shared_d_ff=0),
    "small_segments_padded_bf16": small(tokens=6, hidden=136, num_experts=32, top_k=2,
                                        num_ranks=4, score_fn=0, num_groups=1, topk_groups=1,
                                        capacity_factor=1.0, d_ff=72, shared_d_ff=40,
                                        sel_bias_std=0.0, dispatch_mode=1),
    "softmax_group_limited": small(tokens=700, hidden=136, num_experts=32, top_k=3, num_ranks=8,
                                   score_fn=0, normalize_topk=False, num_groups=8,
                                   topk_groups=2, d_ff=64, shared_d_ff=0, sel_bias_std=0.0),
    "padded_choice_major_round_robin": small(tokens=900, hidden=128, num_experts=24, top_k=3,
                                             num_ranks=7, rank_map=1, score_fn=0,
                                             num_groups=1, topk_groups=1, capacity_factor=0.9,
                                             d_ff=96, shared_d_ff=64, sel_bias_std=0.0,
                                             dispatch_mode=1),
    "padded_f32_small_segments": small(tokens=12, hidden=72, num_experts=16, top_k=2,
                                       num_ranks=4, score_fn=0, num_groups=1, topk_groups=1,
                                       capacity_factor=1.0, d_ff=40, shared_d_ff=0,
                                       act_dtype="f32", sel_bias_std=0.0, dispatch_mode=1),
    # smallest legal sizes: hidden = d_ff = 8 (one 16-byte vector per row)
    "minimal_sizes_bf16": small(tokens=5, hidden=8, num_experts=4, top_k=2, num_ranks=2,
                                num_groups=2, topk_groups=1, d_ff=8, shared_d_ff=8),
    "minimal_sizes_f32": small(tokens=5, hidden=8, num_experts=4, top_k=2, num_ranks=2,
                               score_fn=0, num_groups=1, topk_groups=1, d_ff=8, shared_d_ff=8,
                               act_dtype="f32", sel_bias_std=0.0),
    # at least 512 send rows per expert: the SM-pair (cta_group::2) expert kernels,
    # ragged hidden / d_ff, one expert's rows not a multiple of 256, shared expert
    "pair_kernel_ragged_shared": small(tokens=1500, hidden=264, num_experts=4, top_k=2,
                                       num_ranks=2, num_groups=2, topk_groups=1, d_ff=200,
                                       shared_d_ff=72),
    "pair_kernel_softmax_capacity": small(tokens=2100, hidden=136, num_experts=6, top_k=3,
                                          num_ranks=3, score_fn=0, num_groups=1, topk_groups=1,
                                          capacity_factor=1.1, d_ff=392, shared_d_ff=0,
                                          sel_bias_std=0.0),
    # skewed expert sizes (66, 15, 212, 267 rows) on the 128-row-tile kernels: last
    # tiles of 11 to 84 rows, an expert of one partial tile, a 560-row shared expert
    "skewed_segments_ragged_tails": small(tokens=560, hidden=200, num_experts=4, top_k=1,
                                               num_ranks=2, score_fn=0, num_groups=1,
                                               topk_groups=1, router_offset_std=0.6,
                                               d_ff=136, shared_d_ff=264, sel_bias_std=0.0),
    # 128-row-tile kernels with several row tiles on the busiest experts (skewed routing,
    # about 300 rows per expert), ragged hidden / d_ff, a 1200-row shared expert
    "skewed_multi_tile_segments": small(tokens=1200, hidden=264, num_experts=4, top_k=1,
                                          num_ranks=2, score_fn=0, num_groups=1,
                                          topk_groups=1, router_offset_std=0.8, d_ff=200,
                                          shared_d_ff=72, sel_bias_std=0.0),
    "capacity_exact_boundary": small(tokens=256, hidden=64, num_experts=4, top_k=1, num_ranks=4,
                                     score_fn=0, num_groups=1, topk_groups=1,
                                     capacity_factor=1.0, d_ff=32, shared_d_ff=0,
                                     sel_bias_std=0.0, act_dtype="f32"),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_cases(name):
    w = EDGE[name]
    inp = W.make_inputs(w, seed=3, device="cuda")
    b, _ = run_gpu(w, inp)
    check_layer(w, inp, b)


def test_all_tokens_to_one_expert_with_cap():
    w = EDGE["tiny_capacity_most_dropped"]
    w = dataclasses.replace(w, capacity_factor=1.0)
    inp = W.make_inputs(w, seed=4, device="cuda")
    inp["b_router"][5] += 100.0          # expert 5 is every token's first choice
    b, _ = run_gpu(w, inp)
    r = check_layer(w, inp, b)
    assert host(b.expert_counts)[5] == w.tokens
    assert host(b.kept_counts)[5] == oracle.capacity(w.tokens, w.top_k, w.num_experts, 1.0)


def test_large_selection_bias_forces_choice_but_not_weights():
    w = EDGE["ragged_sigmoid_groups_shared"]
    inp = W.make_inputs(w, seed=5, device="cuda")
    inp["sel_bias"][[1, 2]] = 50.0       # same group: that group and these two experts win
    inp["sel_bias"][[9]] = -50.0         # never chosen
    b, _ = run_gpu(w, inp)
    check_layer(w, inp, b)
    idx = host(b.topk_idx)
    assert np.all(idx[:, 0:2] == [1, 2]) or np.all(np.sort(idx[:, :2], 1) == [1, 2])
    assert not np.any(idx == 9)


def test_layer_replays_from_a_cuda_graph_bit_exactly():
    """The five C-ABI calls can be captured in a CUDA graph; replay gives the same
    bits as direct calls (the benchmark times graph replays)."""
    from expert_routing_router_b300 import moe
    for w in (EDGE["ragged_sigmoid_groups_shared"], W.DSV3_DECODE.with_tokens(8)):
        inp = W.make_inputs(w, seed=2, device="cuda")
        bias0 = inp["sel_bias"].clone()
        b = moe.LayerBuffers(w)
        moe.run_layer(b, inp, bias_step=w.bias_step)
        torch.cuda.synchronize()
        ref_out, ref_bias = b.out.clone(), inp["sel_bias"].clone()
        inp["sel_bias"].copy_(bias0)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            moe.run_layer(b, inp, bias_step=w.bias_step)
        inp["sel_bias"].copy_(bias0)
        b.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(b.out, ref_out)
        assert torch.equal(inp["sel_bias"], ref_bias)
        assert int(b.workspace[:4].view(torch.int32).item()) == 0


# ---------------------------------------------------------------- INT8 all-to-all payload

INT8_EDGE = {
    "int8_ragged_sigmoid_groups_shared": small(payload="int8"),
    "int8_f32_softmax_cap": dataclasses.replace(EDGE["ragged_f32_softmax_cap"], payload="int8"),
    "int8_padded_round_robin": dataclasses.replace(EDGE["padded_choice_major_round_robin"],
                                                   payload="int8"),
    "int8_minimal_sizes": dataclasses.replace(EDGE["minimal_sizes_bf16"], payload="int8"),
    "int8_small_segments": dataclasses.replace(EDGE["small_segments_ragged"], payload="int8"),
    # rows longer than the register-cached part (8192 bf16): the code pass re-reads them
    "int8_long_rows": small(tokens=24, hidden=8200, num_experts=8, top_k=2, num_ranks=2,
                            num_groups=1, topk_groups=1, d_ff=64, shared_d_ff=0,
                            sel_bias_std=0.0, score_fn=0, payload="int8"),
}


@pytest.mark.parametrize("name", list(INT8_EDGE))
def test_int8_payload_cases(name):
    w = INT8_EDGE[name]
    inp = W.make_inputs(w, seed=6, device="cuda")
    b, _ = run_gpu(w, inp)
    check_layer(w, inp, b)


def test_int8_payload_zero_and_extreme_rows():
    """An all-zero token row travels as scale 0 and zero codes; rows scaled by 1e-30
    and 1e3 keep their relative precision (the scale follows the row)."""
    w = INT8_EDGE["int8_ragged_sigmoid_groups_shared"]
    inp = W.make_inputs(w, seed=7, device="cuda")
    inp["x"][0] = 0
    inp["x"][1] *= 1e-30
    inp["x"][2] *= 1e3
    b, _ = run_gpu(w, inp)
    check_layer(w, inp, b)
    slots = host(b.slot_of).reshape(w.tokens, w.top_k)[0]
    for s in slots[slots >= 0]:
        assert float(b.xscale[int(s)]) == 0.0
        assert not b.xperm_q[int(s)].any()


def test_dsv3_prefill_int8_payload(dsv3_inputs):
    w, (inp, hw) = W.DSV3_PREFILL_INT8, dsv3_inputs
    b, bias0 = run_gpu(w, inp)
    check_layer(w, inp, b, n_sample_tokens=1024, n_sample_rows="borders", hw=hw)
    if bias0 is not None:
        inp["sel_bias"].copy_(bias0)
    del b
    torch.cuda.empty_cache()


def test_int8_payload_graph_replay_bit_exact():
    from expert_routing_router_b300 import moe
    w = INT8_EDGE["int8_ragged_sigmoid_groups_shared"]
    inp = W.make_inputs(w, seed=8, device="cuda")
    bias0 = inp["sel_bias"].clone()
    b = moe.LayerBuffers(w)
    moe.run_layer(b, inp, bias_step=w.bias_step)
    torch.cuda.synchronize()
    ref_out, ref_bias = b.out.clone(), inp["sel_bias"].clone()
    inp["sel_bias"].copy_(bias0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.run_layer(b, inp, bias_step=w.bias_step)
    inp["sel_bias"].copy_(bias0)
    b.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(b.out, ref_out)
    assert torch.equal(inp["sel_bias"], ref_bias)
