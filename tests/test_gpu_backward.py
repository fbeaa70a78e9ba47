"""GPU parity of the backward pass: every backward call against the CPU oracle (B300).

Per step the oracle takes the very inputs the GPU step took (the forward's routing,
send rows and expert outputs, the GPU's dyperm / dtopk_w / dlogits), so each
comparison isolates one call:
  combine backward   dyperm (one rounding), dtopk_w (fp32 dot)     4e-3 / 1e-4
  expert FFN dgrad   dxperm rows, dx_shared rows                    2e-2 (bf16 path)
  expert FFN wgrad   dW_gate_up / dW_down of sampled experts and    2e-2
                     hidden units; zeros for experts with no rows   exact
  router backward    dlogits                                        1e-5
                     dx_router, dW_router, db_router                1e-4
  dispatch backward  dx from the GPU's pieces                       one rounding
  end to end         dx from an oracle-only chain (x, weights,      2e-2, and the
                     dout, the GPU's routing)                        delta dx - dout
Tolerances are max-abs normalised (max|got - ref| <= tol * max|ref|).  The full-size
DeepSeek-V3 layer is checked on seeded samples; the small cases in full.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import test_gpu_parity as P
from expert_routing_router_b300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_DW_DOT = 1e-4
TOL_DLOGITS = 1e-5
TOL_ROUTER = 1e-4
TOL_BF16 = 2e-2


def bf16_to_f32(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32)


def rows_of(t, idx):
    return t[torch.as_tensor(np.asarray(idx, np.int64), device=t.device)]


def run_backward(w, inp, seed=0, save=False):
    """Forward then backward; with save=True the forward keeps h and g|u
    (moe_expert_ffn_save) and the backward reuses them instead of recomputing."""
    from expert_routing_router_b300 import moe
    saved = None
    if save:
        b = moe.LayerBuffers(w)
        saved = torch.empty(moe.moe_saved_size(b.cfg), dtype=torch.uint8, device="cuda")
        moe.run_layer(b, inp, saved=saved)
        torch.cuda.synchronize()
        assert int(b.workspace[:4].view(torch.int32).item()) == 0
    else:
        b, _ = P.run_gpu(w, inp)
    g = moe.GradBuffers(w)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1000 + seed)
    dout = torch.randn(w.tokens, w.hidden, generator=gen, device="cuda").to(w.torch_dtype)
    moe.run_layer_backward(b, g, inp, dout, saved=saved)
    torch.cuda.synchronize()
    assert int(g.workspace[:4].view(torch.int32).item()) == 0, "backward status word set"
    return b, g, dout


def check_backward(w, inp, b, g, dout, n_tok=None, n_rows=None, experts=None, n_f=None,
                   seed=0, hw=None):
    if hw is None:
        hw = P.host_weights(inp)
    rng = np.random.default_rng(seed)
    N, d, E, k, F = w.tokens, w.hidden, w.num_experts, w.top_k, w.d_ff
    H = P.host
    x_h, dout_h = H(inp["x"]), H(dout)
    slot_of, topk_w = H(b.slot_of), H(b.topk_w).astype(np.float64)
    idx, logits = H(b.topk_idx), H(b.logits)
    ps = H(b.perm_src)
    kept_rows = np.nonzero(ps >= 0)[0]
    flat_idx = idx.reshape(-1)
    wgu, wd, sgu, sd = hw["w_gate_up"], hw["w_down"], hw["shared_gate_up"], hw["shared_down"]
    toks = np.arange(N, dtype=np.int32) if n_tok is None else np.sort(
        rng.choice(N, size=min(N, n_tok), replace=False)).astype(np.int32)

    # ---- combine backward on the sampled tokens (compact slot numbering)
    sl = slot_of.reshape(N, k)[toks]
    kept_slots = np.unique(sl[sl >= 0])
    remap = np.full(max(int(sl.max()) + 1, 1), -1, np.int64)
    remap[kept_slots] = np.arange(kept_slots.size)
    slc = np.where(sl >= 0, remap[np.maximum(sl, 0)], -1).astype(np.int32)
    y_c = H(rows_of(b.yperm, kept_slots)) if kept_slots.size else np.zeros((0, d), np.uint16)
    dy_ref, dw_ref = oracle.combine_backward(dout_h[toks], y_c, slc, topk_w[toks])
    if kept_slots.size:
        P.close(P.f64(rows_of(g.dyperm, kept_slots)), dy_ref, P.TOL_COMBINE[w.act_dtype],
                "dyperm")
    P.close(H(g.dtopk_w)[toks], dw_ref, TOL_DW_DOT, "dtopk_w")

    # ---- expert FFN dgrad on sampled send rows, shared expert on sampled tokens
    sel = kept_rows if n_rows is None else np.sort(
        rng.choice(kept_rows, size=min(kept_rows.size, n_rows), replace=False))
    if sel.size:
        ref = oracle.ffn_backward_rows(H(rows_of(b.xperm, sel)), H(rows_of(g.dyperm, sel)),
                                       flat_idx[ps[sel]], wgu, wd)
        P.close(P.f64(rows_of(g.dxperm, sel)), ref, TOL_BF16, "dxperm rows")
    if sgu is not None:
        ref = oracle.ffn_backward_rows(x_h[toks], dout_h[toks], np.full(toks.size, E, np.int32),
                                       wgu, wd, sgu, sd)
        P.close(P.f64(rows_of(g.dx_shared, toks)), ref, TOL_BF16, "dx_shared rows")

    # ---- expert FFN wgrad
    kept_counts, starts = H(b.kept_counts), H(b.expert_start)
    if experts is None:
        experts = list(range(E))
    fs = None if n_f is None else np.sort(rng.choice(F, size=min(F, n_f), replace=False))
    for e in experts:
        n = int(kept_counts[e])
        if n == 0:
            assert not g.dw_gate_up[e].any() and not g.dw_down[e].any(), f"expert {e} not zero"
            continue
        r = np.arange(starts[e], starts[e] + n)
        cd, rg, ru = oracle.ffn_wgrad(H(rows_of(b.xperm, r)), H(rows_of(g.dyperm, r)), wgu[e],
                                      wd[e], fs)
        f_idx = np.arange(F) if fs is None else fs
        got_wd = P.f64(g.dw_down[e])[:, f_idx].T
        got_wgu = P.f64(g.dw_gate_up[e])
        P.close(got_wd, cd, TOL_BF16, f"dW_down[{e}]")
        P.close(got_wgu[f_idx], rg, TOL_BF16, f"dW_gate[{e}]")
        P.close(got_wgu[F + f_idx], ru, TOL_BF16, f"dW_up[{e}]")
    if sgu is not None:
        Fs = w.shared_d_ff
        fss = None if n_f is None else np.sort(rng.choice(Fs, size=min(Fs, n_f), replace=False))
        cd, rg, ru = oracle.ffn_wgrad(x_h, dout_h, sgu, sd, fss)
        f_idx = np.arange(Fs) if fss is None else fss
        P.close(P.f64(g.dshared_down)[:, f_idx].T, cd, TOL_BF16, "dW_shared_down")
        got = P.f64(g.dshared_gate_up)
        P.close(got[f_idx], rg, TOL_BF16, "dW_shared_gate")
        P.close(got[Fs + f_idx], ru, TOL_BF16, "dW_shared_up")

    # ---- router backward from the GPU's dtopk_w, then its parameter and input grads
    dl_ref = oracle.route_backward(logits, idx, H(g.dtopk_w).astype(np.float64), w.score_fn,
                                   w.normalize_topk)
    dl_gpu = H(g.dlogits)
    P.close(dl_gpu, dl_ref, TOL_DLOGITS, "dlogits")
    dxr_ref, dwr_ref, db_ref = oracle.router_grads(x_h, H(inp["w_router"]),
                                                   dl_gpu.astype(np.float64), toks)
    P.close(H(g.dx_router)[toks], dxr_ref, TOL_ROUTER, "dx_router")
    P.close(H(g.dw_router), dwr_ref, TOL_ROUTER, "dW_router")
    P.close(H(g.db_router), db_ref, TOL_ROUTER, "db_router")

    # ---- dispatch backward from the GPU's pieces
    ref = oracle.dispatch_backward(toks, dout_h, H(g.dxperm), slot_of,
                                   None if g.dx_shared is None else H(g.dx_shared),
                                   H(g.dx_router))
    dx_got = P.f64(g.dx)
    P.close(dx_got[toks], ref, P.TOL_COMBINE[w.act_dtype], "dx (dispatch backward)")

    # ---- end to end: dx from an oracle-only chain (GPU routing, oracle everything else)
    e2e = np.zeros((toks.size, d))
    dw_e2e = np.zeros((toks.size, k))
    pairs = [(i, j) for i, t in enumerate(toks) for j in range(k) if slot_of[t * k + j] >= 0]
    if pairs:
        pi = np.array([p_[0] for p_ in pairs])
        pj = np.array([p_[1] for p_ in pairs])
        pt = toks[pi]
        pe = idx[pt, pj].astype(np.int32)
        xr = np.ascontiguousarray(x_h[pt])
        y = oracle.expert_rows(xr, pe, wgu, wd)                      # fp64, all pairs at once
        g32 = bf16_to_f32(dout_h[pt]).astype(np.float64)
        dw_e2e[pi, pj] = np.einsum("rd,rd->r", g32, y)
        dy = oracle.float_to_bf16((topk_w[pt, pj][:, None] * g32).astype(np.float32))
        dxr_rows = oracle.ffn_backward_rows(xr, dy, pe, wgu, wd)
        np.add.at(e2e, pi, dxr_rows)
    dl_e2e = oracle.route_backward(logits[toks], idx[toks], dw_e2e, w.score_fn,
                                   w.normalize_topk)
    x_sub = np.ascontiguousarray(x_h[toks])
    e2e += oracle.router_grads(x_sub, H(inp["w_router"]), dl_e2e, params=False)[0]
    if sgu is not None:
        e2e += oracle.ffn_backward_rows(x_h[toks], dout_h[toks], np.full(toks.size, E, np.int32),
                                        wgu, wd, sgu, sd)
    g_in = bf16_to_f32(dout_h[toks]).astype(np.float64)
    ref = g_in + e2e
    P.close(dx_got[toks], ref, TOL_BF16, "dx end to end")
    allow = TOL_BF16 * np.max(np.abs(e2e)) + P.OUT_ROUNDING[w.act_dtype] * np.abs(ref)
    assert np.all(np.abs((dx_got[toks] - g_in) - e2e) <= allow), "dx - dout end to end"


BWD_EDGE = {
    "sigmoid_groups_shared": P.small(),
    "softmax_unnorm_capacity": P.small(tokens=777, hidden=136, num_experts=12, top_k=3,
                                       num_ranks=3, score_fn=0, normalize_topk=False,
                                       num_groups=1, topk_groups=1, capacity_factor=1.0,
                                       d_ff=40, shared_d_ff=0, sel_bias_std=0.0),
    "softmax_norm_padded": dataclasses.replace(P.EDGE["padded_choice_major_round_robin"]),
    "small_segments": P.EDGE["small_segments_ragged"],
    "minimal_sizes": P.EDGE["minimal_sizes_bf16"],
    "long_segments": P.small(tokens=3000, hidden=192, num_experts=4, top_k=2, num_ranks=2,
                             score_fn=0, num_groups=1, topk_groups=1, d_ff=136, shared_d_ff=64,
                             sel_bias_std=0.0),
}


@pytest.mark.parametrize("name", list(BWD_EDGE))
def test_backward_cases(name):
    w = BWD_EDGE[name]
    inp = W.make_inputs(w, seed=21, device="cuda")
    b, g, dout = run_backward(w, inp)
    check_backward(w, inp, b, g, dout, n_tok=None if w.tokens <= 1000 else 96)


def test_backward_dsv3_prefill(dsv3_inputs):
    w, (inp, hw) = W.DSV3_PREFILL, dsv3_inputs
    b, g, dout = run_backward(w, inp)
    counts = P.host(b.kept_counts)
    nz = np.nonzero(counts)[0]
    small_e = [int(e) for e in nz[np.argsort(counts[nz])[:2]]]
    zero_e = [int(e) for e in np.nonzero(counts == 0)[0][:1]]
    check_backward(w, inp, b, g, dout, n_tok=8, n_rows=24, experts=small_e + zero_e, n_f=6,
                   hw=hw)
    del b, g
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def dsv3_inputs():
    inp = W.make_inputs(W.DSV3_PREFILL, seed=0, device="cuda")
    yield inp, P.host_weights(inp)
    del inp
    torch.cuda.empty_cache()


def test_backward_graph_replay_bit_exact():
    from expert_routing_router_b300 import moe
    w = BWD_EDGE["sigmoid_groups_shared"]
    inp = W.make_inputs(w, seed=22, device="cuda")
    b, g, dout = run_backward(w, inp)
    ref = [t.clone() for t in (g.dx, g.dw_gate_up, g.dw_down, g.dw_router)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        moe.run_layer_backward(b, g, inp, dout)
    g.dx.zero_()
    g.dw_gate_up.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for a, r in zip((g.dx, g.dw_gate_up, g.dw_down, g.dw_router), ref):
        assert torch.equal(a, r)


@pytest.mark.parametrize("name", ["sigmoid_groups_shared", "long_segments", "softmax_norm_padded"])
def test_backward_with_saved_activations(name):
    """Training forward (moe_expert_ffn_save) + backward reusing its h and g|u: full
    parity, and the same gradients as the recomputing backward (same kernels, same
    accumulation order)."""
    w = BWD_EDGE[name]
    inp = W.make_inputs(w, seed=23, device="cuda")
    b, g, dout = run_backward(w, inp, save=True)
    check_backward(w, inp, b, g, dout, n_tok=None if w.tokens <= 1000 else 96)
    b2, g2, dout2 = run_backward(w, inp, save=False)
    assert torch.equal(dout, dout2)
    for name_ in ("dx", "dw_gate_up", "dw_down", "dxperm"):
        a, r = getattr(g, name_), getattr(g2, name_)
        if name_ == "dxperm":
            rows = torch.from_numpy(np.nonzero(P.host(b.perm_src) >= 0)[0]).cuda()
            a, r = a[rows], r[rows]
        assert torch.equal(a, r), name_


def test_backward_dsv3_prefill_saved(dsv3_inputs):
    w, (inp, hw) = W.DSV3_PREFILL, dsv3_inputs
    b, g, dout = run_backward(w, inp, save=True)
    counts = P.host(b.kept_counts)
    nz = np.nonzero(counts)[0]
    check_backward(w, inp, b, g, dout, n_tok=8, n_rows=24,
                   experts=[int(nz[np.argmax(counts[nz])])], n_f=4, hw=hw)
    del b, g
    torch.cuda.empty_cache()
