"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks one oracle function against what the pages print, a closed form,
an invariant, a library routine on a special case, or brute force on tiny inputs.
The cases are chosen so that a plausible slip (a dropped term, a wrong sign, a
swapped gate/up, a transposed operand, an off-by-one in the cap) fails at least one.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from expert_routing_router_b300 import workloads as W


def f32_ulp(x):
    x = np.abs(np.asarray(x, dtype=np.float32))
    return np.spacing(x).astype(np.float64)


# ------------------------------------------------------------------ worked example

def test_worked_example_counts_match_page(golden):
    """Glossary page's routing example: counts within the printed range."""
    g = golden("worked_example_tiny_top2.txt")
    inp = W.make_inputs(W.TINY_TOP2_F32, seed=0, with_experts=False)
    logits = oracle.router_logits(inp["x"].numpy(), inp["w_router"].numpy(),
                                  inp["b_router"].numpy())
    idx, _ = oracle.route(logits, 2, score_fn=0, normalize=True)
    d = oracle.dispatch(idx, E=8, R=4, rank_map=0, cf=0.0)
    ec, rc = d["expert_counts"], d["rank_counts"]
    assert ec.sum() == g["assignments"] == rc.sum()
    assert ec.sum() / 8 == g["expert_count_mean"]
    assert ec.min() == g["expert_count_min"] and ec.max() == g["expert_count_max"]
    assert rc.min() == g["rank_count_min"] and rc.max() == g["rank_count_max"]


def test_worked_example_matches_torch_topk_library():
    """Same workload: oracle selection == torch.topk of torch's own fp32 router output."""
    inp = W.make_inputs(W.TINY_TOP2_F32, seed=0, with_experts=False)
    with torch.no_grad():
        t_logits = inp["x"] @ inp["w_router"].T + inp["b_router"]
        _, t_idx = t_logits.topk(2, dim=-1)
    logits = oracle.router_logits(inp["x"].numpy(), inp["w_router"].numpy(),
                                  inp["b_router"].numpy())
    # fp32-accurate logits: within a few fp32 ulps of torch's fp32 GEMM
    assert np.max(np.abs(logits - t_logits.numpy())) < 4e-6
    idx, _ = oracle.route(logits, 2, score_fn=0)
    np.testing.assert_array_equal(idx, t_idx.numpy())


# ------------------------------------------------------------------ router logits

def test_router_logits_vs_fp64_library_matmul():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((37, 40)).astype(np.float32)
    w = rng.uniform(-0.2, 0.2, (11, 40)).astype(np.float32)
    b = rng.uniform(-0.2, 0.2, 11).astype(np.float32)
    got = oracle.router_logits(x, w, b)
    ref = (torch.from_numpy(x).double() @ torch.from_numpy(w).double().T
           + torch.from_numpy(b).double()).numpy()
    assert np.all(np.abs(got - ref) <= 0.5 * f32_ulp(ref) * 1.0001 + 1e-30)
    # bias really is added (not dropped): removing it moves the result
    got_nb = oracle.router_logits(x, w, None)
    assert np.max(np.abs(got - got_nb - b[None, :])) < 1e-5


def test_router_logits_bf16_input_exact_widening():
    rng = np.random.default_rng(2)
    xt = torch.from_numpy(rng.standard_normal((9, 16)).astype(np.float32)).bfloat16()
    bits = xt.view(torch.int16).numpy().view(np.uint16)
    w = rng.uniform(-1, 1, (5, 16)).astype(np.float32)
    got = oracle.router_logits(bits, w)
    ref = (xt.double() @ torch.from_numpy(w).double().T).numpy()
    assert np.all(np.abs(got - ref) <= 0.5 * f32_ulp(ref) * 1.0001 + 1e-30)


# ------------------------------------------------------------------ sigmoid spec

def test_sigmoid_spec_error_bound_and_fixed_points():
    l = np.concatenate([np.linspace(-90, 30, 400001, dtype=np.float32),
                        np.random.default_rng(3).standard_normal(200000).astype(np.float32) * 4])
    s = oracle.sigmoid_spec(l)
    exact = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
    ulps = np.abs(s - exact) / f32_ulp(exact)
    inside = (l > -86) & (l < 20)
    assert ulps[inside].max() <= 3.0, ulps[inside].max()
    assert oracle.sigmoid_spec(np.float32([0.0]))[0] == 0.5
    assert np.all(oracle.sigmoid_spec(np.float32([20.0, 25.0, 1e30])) == 1.0)
    # monotone non-decreasing along the sweep
    sw = s[:400001]
    assert np.all(np.diff(sw) >= 0)
    # symmetry S(-l) = 1 - S(l) within the bound
    z = np.linspace(-15, 15, 3001, dtype=np.float32)
    assert np.max(np.abs(oracle.sigmoid_spec(z) + oracle.sigmoid_spec(-z) - 1.0)) < 3e-7


# ------------------------------------------------------------------ softmax routing

@pytest.mark.parametrize("k", [1, 2, 5])
def test_softmax_topk_vs_torch_topk_and_softmax(k):
    rng = np.random.default_rng(10 + k)
    logits = rng.standard_normal((300, 13)).astype(np.float32) * 3
    for normalize in (False, True):
        idx, w = oracle.route(logits, k, score_fn=0, normalize=normalize)
        tl = torch.from_numpy(logits)
        _, tidx = tl.topk(k, dim=-1)
        np.testing.assert_array_equal(idx, tidx.numpy())
        p = torch.softmax(tl.double(), dim=-1).gather(1, tidx.long())
        if normalize:
            p = p / p.sum(-1, keepdim=True)
        np.testing.assert_allclose(w, p.numpy(), rtol=1e-12, atol=0)


def test_softmax_top1_two_experts_closed_form():
    l = np.array([[2.0, -1.0], [0.25, 0.75]], dtype=np.float32)
    idx, w = oracle.route(l, 1, score_fn=0, normalize=False)
    assert idx.tolist() == [[0], [1]]
    np.testing.assert_allclose(w[:, 0], [1 / (1 + math.exp(-3.0)), 1 / (1 + math.exp(-0.5))],
                               rtol=1e-14)


def _brute_topk(keys, k, allowed=None):
    """The unique k-subset S with every member ranking before every non-member
    (larger key, or equal key and lower index), found by enumerating all subsets."""
    E = len(keys)
    pool = [e for e in range(E) if allowed is None or allowed[e]]
    found = []
    for S in itertools.combinations(pool, k):
        rest = [f for f in pool if f not in S]
        if all(keys[e] > keys[f] or (keys[e] == keys[f] and e < f) for e in S for f in rest):
            found.append(S)
    assert len(found) == 1
    S = found[0]
    return sorted(S, key=lambda e: (-keys[e], e))


def test_topk_ties_bruteforce():
    rng = np.random.default_rng(4)
    logits = rng.integers(-2, 3, size=(200, 6)).astype(np.float32)  # many ties
    for k in (1, 2, 3, 6):
        idx, _ = oracle.route(logits, k, score_fn=0)
        for t in range(logits.shape[0]):
            assert list(idx[t]) == _brute_topk(list(logits[t]), k)


# ------------------------------------------------------------------ sigmoid + groups

def _brute_group_route(l, bias, k, G, TG):
    E = len(l)
    gs = E // G
    s = oracle.sigmoid_spec(np.asarray(l, np.float32))
    key = (s + np.asarray(bias, np.float32)).astype(np.float32)
    # group score: the largest fp32 pair sum inside the group (= sum of the top two)
    gsc = []
    for g in range(G):
        mem = range(g * gs, (g + 1) * gs)
        if gs == 1:
            gsc.append(key[g * gs])
        else:
            gsc.append(max(np.float32(key[a] + key[b]) for a, b in itertools.combinations(mem, 2)))
    kept = _brute_topk(gsc, TG)
    allowed = [(e // gs) in kept for e in range(E)]
    sel = _brute_topk(list(key), k, allowed)
    return sel, s


@pytest.mark.parametrize("E,G,TG,k", [(8, 4, 2, 2), (8, 4, 1, 2), (12, 3, 2, 4), (8, 8, 3, 3),
                                      (16, 4, 2, 8), (6, 1, 1, 3)])
def test_group_limited_sigmoid_bruteforce(E, G, TG, k):
    rng = np.random.default_rng(E * 100 + G * 10 + k)
    N = 150
    logits = (rng.standard_normal((N, E)) * 2).astype(np.float32)
    logits[:20] = np.round(logits[:20])  # ties in sigmoid values too
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    bias[: E // 2] = np.round(bias[: E // 2], 1)
    idx, w = oracle.route(logits, k, score_fn=1, normalize=True, num_groups=G, topk_groups=TG,
                          sel_bias=bias)
    for t in range(N):
        sel, s = _brute_group_route(logits[t], bias, k, G, TG)
        assert list(idx[t]) == sel, t
        assert len({e // (E // G) for e in idx[t]}) <= TG
        sv = s[idx[t]].astype(np.float64)
        np.testing.assert_allclose(w[t], sv / sv.sum(), rtol=1e-14)


def test_bias_is_selection_only():
    rng = np.random.default_rng(5)
    E, k, N = 16, 4, 64
    logits = rng.standard_normal((N, E)).astype(np.float32)
    forced = [3, 7, 11, 12]
    bias = np.zeros(E, np.float32)
    bias[forced] = 50.0
    idx, w = oracle.route(logits, k, score_fn=1, normalize=True, sel_bias=bias)
    s = 1.0 / (1.0 + np.exp(-logits.astype(np.float64)))
    for t in range(N):
        assert sorted(idx[t]) == forced
        sv = s[t, idx[t]]
        np.testing.assert_allclose(w[t], sv / sv.sum(), rtol=1e-6)
    # a different bias that leaves the selection unchanged leaves weights bit-identical
    bias2 = bias.copy()
    bias2[forced] = 80.0
    bias2[0] = -3.0
    idx2, w2 = oracle.route(logits, k, score_fn=1, normalize=True, sel_bias=bias2)
    np.testing.assert_array_equal(idx2, idx)
    np.testing.assert_array_equal(w2, w)


def test_unnormalized_sigmoid_weights_are_scores():
    l = np.array([[0.0, 1.0, -1.0, 2.0]], np.float32)
    idx, w = oracle.route(l, 2, score_fn=1, normalize=False)
    assert idx.tolist() == [[3, 1]]
    np.testing.assert_allclose(w[0], [1 / (1 + math.exp(-2)), 1 / (1 + math.exp(-1))], rtol=1e-6)


# ------------------------------------------------------------------ capacity + dispatch

def test_capacity_closed_form():
    assert oracle.capacity(16384, 1, 32, 1.25) == 640
    assert oracle.capacity(32768, 2, 64, 1.25) == 1280
    assert oracle.capacity(10, 1, 4, 1.0) == 3          # ceil(2.5)
    assert oracle.capacity(8, 1, 4, 1.0) == 2           # exact, no round-up
    assert oracle.capacity(8, 2, 4, 0.0) > 10 ** 9      # no cap


def _check_dispatch(idx, E, R, rank_map, cf, d):
    N, k = idx.shape
    A = N * k
    flat = idx.reshape(-1)
    C = oracle.capacity(N, k, E, cf)
    # counts: bincount, sum N*k
    np.testing.assert_array_equal(d["expert_counts"], np.bincount(flat, minlength=E))
    assert d["expert_counts"].sum() == A
    np.testing.assert_array_equal(d["kept_counts"], np.minimum(d["expert_counts"], C))
    # brute force keep rule: kept iff fewer than C earlier assignments to that expert
    kept = np.array([np.count_nonzero(flat[:a] == flat[a]) < C for a in range(A)])
    np.testing.assert_array_equal(d["slot_of"] >= 0, kept)
    # rank map and per-rank sums
    ranks = np.array([(e % R) if rank_map else e // (E // R) for e in range(E)])
    for r in range(R):
        assert d["rank_counts"][r] == d["kept_counts"][ranks == r].sum()
    np.testing.assert_array_equal(d["rank_offsets"], np.concatenate([[0], np.cumsum(d["rank_counts"])]))
    assert d["num_kept"] == d["kept_counts"].sum() == kept.sum()
    # slot_of / perm_src are inverse bijections on kept assignments
    nk = d["num_kept"]
    ps = d["perm_src"]
    assert np.all(ps[nk:] == -1)
    assert sorted(ps[:nk].tolist()) == sorted(np.nonzero(kept)[0].tolist())
    for s in range(nk):
        assert d["slot_of"][ps[s]] == s
    # send order: (rank, expert, token order)
    keyv = [(ranks[flat[a]], flat[a], a) for a in ps[:nk]]
    assert keyv == sorted(keyv)
    for e in range(E):
        rows = [s for s in range(nk) if flat[ps[s]] == e]
        if rows:
            assert rows[0] == d["expert_start"][e] and len(rows) == d["kept_counts"][e]


@pytest.mark.parametrize("N,E,k,R,rank_map,cf", [
    (40, 4, 1, 2, 0, 1.0), (37, 8, 2, 4, 0, 1.25), (50, 6, 3, 3, 1, 0.8), (25, 5, 2, 5, 0, 0.0),
    (64, 16, 4, 5, 1, 1.0), (10, 3, 3, 1, 0, 0.3)])
def test_dispatch_invariants_and_bruteforce(N, E, k, R, rank_map, cf):
    rng = np.random.default_rng(N + E + k)
    # skewed choices (hot experts) so that caps bite
    p = rng.dirichlet(np.ones(E) * 0.5)
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(N)]).astype(np.int32)
    d = oracle.dispatch(idx, E, R, rank_map, cf)
    _check_dispatch(idx, E, R, rank_map, cf, d)


def test_dispatch_all_to_one_expert_and_all_dropped():
    N, E, k = 30, 4, 1
    idx = np.full((N, k), 2, np.int32)
    d = oracle.dispatch(idx, E, 2, 0, 1.0)      # C = ceil(30/4) = 8
    assert d["kept_counts"].tolist() == [0, 0, 8, 0]
    assert (d["slot_of"] >= 0).sum() == 8 and np.all(d["slot_of"][:8] == np.arange(8))
    d = oracle.dispatch(idx, E, 2, 0, 0.0001)   # C = 1
    assert d["num_kept"] == 1 and d["slot_of"][0] == 0 and np.all(d["slot_of"][1:] == -1)


def test_rank_map_matches_page_example():
    # glossary example: experts 0-1 on GPU 0, 2-3 on GPU 1, ... (e // 2 for 8 experts on 4)
    assert [oracle.rank_of(e, 8, 4, 0) for e in range(8)] == [0, 0, 1, 1, 2, 2, 3, 3]
    assert [oracle.rank_of(e, 256, 40, 1) for e in (0, 39, 40, 255)] == [0, 39, 0, 15]


# ------------------------------------------------------------------ expert FFN + combine

def _torch_swiglu(x, wgu, wd):
    F = wgu.shape[0] // 2
    g = torch.nn.functional.linear(x, wgu[:F])
    u = torch.nn.functional.linear(x, wgu[F:])
    return torch.nn.functional.linear(torch.nn.functional.silu(g) * u, wd)


def test_single_expert_layer_is_dense_swiglu():
    """E=1, k=1, no cap: the layer reduces to x + SwiGLU(x) (torch fp64 library ops)."""
    rng = np.random.default_rng(6)
    N, d, F = 23, 24, 16
    x = rng.standard_normal((N, d)).astype(np.float32)
    wgu = (rng.standard_normal((1, 2 * F, d)) * 0.3).astype(np.float32)
    wd = (rng.standard_normal((1, d, F)) * 0.3).astype(np.float32)
    idx = np.zeros((N, 1), np.int32)
    w = np.ones((N, 1))
    disp = oracle.dispatch(idx, 1, 1, 0, 0.0)
    out = oracle.layer_tokens(np.arange(N), x, idx, w, disp["slot_of"], wgu, wd)
    ref = torch.from_numpy(x).double() + _torch_swiglu(
        torch.from_numpy(x).double(), torch.from_numpy(wgu[0]).double(),
        torch.from_numpy(wd[0]).double())
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    y = oracle.expert_rows(x, np.zeros(N, np.int32), wgu, wd)
    np.testing.assert_allclose(y, (ref - torch.from_numpy(x).double()).numpy(), rtol=1e-12,
                               atol=1e-12)


def test_shared_expert_rows_bf16():
    rng = np.random.default_rng(7)
    N, d, F, Fs = 5, 16, 8, 24
    to_bits = lambda a: torch.from_numpy(a).bfloat16().view(torch.int16).numpy().view(np.uint16)
    x = to_bits(rng.standard_normal((N, d)).astype(np.float32))
    wgu = to_bits((rng.standard_normal((2, 2 * F, d)) * 0.2).astype(np.float32))
    wd = to_bits((rng.standard_normal((2, d, F)) * 0.2).astype(np.float32))
    sgu = to_bits((rng.standard_normal((2 * Fs, d)) * 0.2).astype(np.float32))
    sd = to_bits((rng.standard_normal((d, Fs)) * 0.2).astype(np.float32))
    bf = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double()
    y = oracle.expert_rows(x, np.array([2, 1, 0, 2, 1], np.int32), wgu, wd, sgu, sd)
    ref_s = _torch_swiglu(bf(x), bf(sgu), bf(sd)).numpy()
    ref_1 = _torch_swiglu(bf(x), bf(wgu)[1], bf(wd)[1]).numpy()
    ref_0 = _torch_swiglu(bf(x), bf(wgu)[0], bf(wd)[0]).numpy()
    np.testing.assert_allclose(y[[0, 3]], ref_s[[0, 3]], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(y[[1, 4]], ref_1[[1, 4]], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(y[2], ref_0[2], rtol=1e-12, atol=1e-13)


def test_identical_experts_full_topk_gives_x_plus_ffn():
    """k = E, normalised softmax weights, identical experts: out = x + FFN(x)."""
    rng = np.random.default_rng(8)
    N, d, F, E = 19, 16, 8, 4
    x = rng.standard_normal((N, d)).astype(np.float32)
    g = (rng.standard_normal((2 * F, d)) * 0.3).astype(np.float32)
    dn = (rng.standard_normal((d, F)) * 0.3).astype(np.float32)
    wgu = np.stack([g] * E)
    wd = np.stack([dn] * E)
    logits = rng.standard_normal((N, E)).astype(np.float32)
    idx, w = oracle.route(logits, E, score_fn=0, normalize=True)
    disp = oracle.dispatch(idx, E, 2, 0, 0.0)
    out = oracle.layer_tokens(np.arange(N), x, idx, w, disp["slot_of"], wgu, wd)
    xd = torch.from_numpy(x).double()
    ref = xd + _torch_swiglu(xd, torch.from_numpy(g).double(), torch.from_numpy(dn).double())
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    # the permuted-buffer path gives the same numbers: combine(yperm) == layer
    xperm = x[disp["perm_src"][:disp["num_kept"]] // E]
    yperm = oracle.expert_rows(xperm, idx.reshape(-1)[disp["perm_src"][:disp["num_kept"]]], wgu, wd)
    out2 = oracle.combine(np.arange(N), x, yperm.astype(np.float32), disp["slot_of"], w)
    np.testing.assert_allclose(out2, ref.numpy(), rtol=1e-6, atol=1e-6)


def test_combine_weights_closed_form_and_fully_dropped_is_residual():
    N, d, k = 3, 4, 2
    x = np.arange(N * d, dtype=np.float32).reshape(N, d) - 5
    yperm = np.array([[1, 1, 1, 1], [10, 20, 30, 40], [0, 0, 0, 2]], np.float32)
    slot_of = np.array([0, 1, 2, -1, -1, -1], np.int32)      # token 2 fully dropped
    w = np.array([[0.25, 0.5], [2.0, 7.0], [1.0, 1.0]])
    out = oracle.combine(np.arange(N), x, yperm, slot_of, w)
    np.testing.assert_array_equal(out[0], x[0] + 0.25 * yperm[0] + 0.5 * yperm[1])
    np.testing.assert_array_equal(out[1], x[1] + 2.0 * yperm[2])
    np.testing.assert_array_equal(out[2], x[2])
    ys = np.full((N, d), 0.5, np.float32)
    out = oracle.combine(np.arange(N), x, yperm, slot_of, w, ys)
    np.testing.assert_array_equal(out[2], x[2] + 0.5)


# ------------------------------------------------------------------ bias update

def test_bias_update_sign_rule():
    E, N, k = 4, 6, 2                 # mean load N*k/E = 3
    counts = np.array([5, 3, 0, 4], np.int32)
    b0 = np.array([0.1, -0.2, 0.0, 1e-3], np.float32)
    b1 = oracle.bias_update(counts, b0, N, k, 1e-3)
    step = np.float32(1e-3)
    assert b1[0] == np.float32(b0[0] - step)      # overloaded: lowered
    assert b1[1] == b0[1]                         # at the mean: unchanged
    assert b1[2] == np.float32(b0[2] + step)      # underloaded: raised
    assert b1[3] == np.float32(b0[3] - step) == 0.0
    # fractional mean (N*k/E = 2.5): 3 is above, 2 below
    b2 = oracle.bias_update(np.array([3, 2, 2, 3], np.int32), np.zeros(4, np.float32), 5, 2, 0.5)
    assert b2.tolist() == [-0.5, 0.5, 0.5, -0.5]


# ------------------------------------------------------------------ capacity-padded, choice-major

def test_choice_major_priority_worked_example():
    """3 tokens, 2 experts, top-2, C = 2.  Token order drops token 2's first choice
    (expert 1 is full with tokens 0 and 1's second choices); choice-major priority
    (all first choices first) keeps it and drops token 1's second choice instead."""
    idx = np.array([[0, 1], [0, 1], [1, 0]], np.int32)
    cf = 0.6                                        # C = ceil(0.6 * 3 * 2 / 2) = 2
    d0 = oracle.dispatch(idx, 2, 1, 0, cf, mode=0)
    d1 = oracle.dispatch(idx, 2, 1, 0, cf, mode=1)
    assert d0["capacity"] == d1["capacity"] == 2
    assert (d0["slot_of"].reshape(3, 2) >= 0).tolist() == [[True, True], [True, True],
                                                          [False, False]]
    assert (d1["slot_of"].reshape(3, 2) >= 0).tolist() == [[True, True], [True, False],
                                                          [True, False]]
    # padded layout: expert e's rows start at e * C; token 2's first choice is row 0 of
    # expert 1 (it came first in priority order), token 0's second choice row 1
    assert d1["expert_start"].tolist() == [0, 2]
    assert d1["slot_of"].tolist() == [0, 3, 1, -1, 2, -1]
    assert d1["perm_src"].tolist() == [0, 2, 4, 1]


@pytest.mark.parametrize("N,E,k,R,rank_map,cf", [
    (40, 4, 2, 2, 0, 1.0), (37, 8, 3, 4, 0, 0.7), (50, 6, 2, 3, 1, 1.25), (64, 16, 4, 5, 1, 0.5)])
def test_choice_major_padded_dispatch_bruteforce(N, E, k, R, rank_map, cf):
    rng = np.random.default_rng(N * 7 + E)
    p = rng.dirichlet(np.ones(E) * 0.5)
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(N)]).astype(np.int32)
    d = oracle.dispatch(idx, E, R, rank_map, cf, mode=1)
    C = d["capacity"]
    flat = idx.reshape(-1)
    order = [t * k + j for j in range(k) for t in range(N)]   # choice-major priority
    rank_in = {}
    kept = np.zeros(N * k, bool)
    pos = np.zeros(N * k, int)
    for a in order:
        e = flat[a]
        before = rank_in.get(e, 0)
        pos[a] = before
        kept[a] = before < C
        rank_in[e] = before + 1
    np.testing.assert_array_equal(d["expert_counts"], np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(d["kept_counts"], np.minimum(d["expert_counts"], C))
    np.testing.assert_array_equal(d["slot_of"] >= 0, kept)
    ranks = np.array([(e % R) if rank_map else e // (E // R) for e in range(E)])
    send = sorted(range(E), key=lambda e: (ranks[e], e))
    for sp, e in enumerate(send):
        assert d["expert_start"][e] == sp * C
    for a in np.nonzero(kept)[0]:
        assert d["slot_of"][a] == d["expert_start"][flat[a]] + pos[a]
    assert d["send_rows"] == E * C and d["perm_src"].size == E * C
    for s in range(E * C):
        a = d["perm_src"][s]
        if a >= 0:
            assert d["slot_of"][a] == s
    assert (d["perm_src"] >= 0).sum() == kept.sum() == d["num_kept"]
    first = [send.index(e) for e in range(E)]
    for r in range(R):
        assert d["rank_counts"][r] == d["kept_counts"][ranks == r].sum()
        assert d["rank_offsets"][r] == min(first[e] for e in range(E) if ranks[e] == r) * C
    assert d["rank_offsets"][R] == E * C


# ------------------------------------------------------------------ INT8 payload

def _bf16_bits(a):
    return torch.tensor(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def test_q8_codes_closed_form():
    """Rows whose scale and its reciprocal are exact (max 127 -> s = 1, max 254 -> s = 2,
    1/s = 0.5): every code is v / s rounded half to even, clamped; a zero row has scale
    0 and zero codes."""
    rows = np.array([[127, -63.5, 31.75, 0, 0.5, -127, 1.5, 2.5, -0.5, 3.49],
                     [254, 3, 5, -7, 1, -1, 0, 9, 11, -254],
                     [0] * 10], np.float32)
    want_q = np.array([[127, -64, 32, 0, 0, -127, 2, 2, 0, 3],
                       [127, 2, 2, -4, 0, 0, 0, 4, 6, -127],
                       [0] * 10], np.int8)
    want_s = np.array([1.0, 2.0, 0.0], np.float32)
    for arr in (rows, _bf16_bits(rows[:, :8])):
        q, s = oracle.quant_rows(arr)
        np.testing.assert_array_equal(q, want_q[:, :arr.shape[1]])
        np.testing.assert_array_equal(s, want_s)


def test_q8_error_bound_and_extremes():
    """|(float)q*s - v| <= s/2 plus rounding: v*r with r = fl(1/s) is within 3 units
    of 2^-24 relative of v/s (so within 127 * 3 * 2^-24 < 2^-15 of a code unit), and the
    product q*s adds 2^-24 relative; each nonzero row reaches +-127 at its largest
    magnitude; codes keep the sign of v."""
    rng = np.random.default_rng(5)
    rows = (rng.standard_normal((64, 200)) *
            np.exp(rng.uniform(-20, 20, size=(64, 1)))).astype(np.float32)
    rows[3] = 0.0
    rows[4, :] = 1e-30                       # tiny, denormal-free scale
    q, s = oracle.quant_rows(rows)
    deq = oracle.dequant_rows(q, s, "f32").astype(np.float64)
    bound = s.astype(np.float64)[:, None] * (0.5 + 2.0 ** -15)
    assert np.all(np.abs(deq - rows) <= bound)
    for r in range(64):
        if s[r] == 0:
            assert not q[r].any()
            continue
        am = int(np.argmax(np.abs(rows[r])))
        assert abs(int(q[r, am])) == 127
    assert np.all((q == 0) | (np.sign(q) == np.sign(rows)))
    assert np.abs(q.astype(np.int32)).max() <= 127


def test_q8_skips_invalid_rows():
    rows = np.ones((3, 8), np.float32)
    q, s = oracle.quant_rows(rows, valid=np.array([0, -1, 5], np.int32))
    assert np.isnan(s[1]) and not q[1].any()
    assert s[0] == s[2] == np.float32(1.0) / np.float32(127.0)


def test_float_to_bf16_matches_torch():
    """The oracle's fp32 -> bf16 rounding against torch's conversion (round to nearest
    even), including exact ties and values just either side of them."""
    rng = np.random.default_rng(6)
    base = rng.standard_normal(4096).astype(np.float32) * 100
    bits = base.view(np.uint32) & 0xffff0000
    ties = (bits | 0x8000).view(np.float32)
    below = (bits | 0x7fff).view(np.float32)
    above = (bits | 0x8001).view(np.float32)
    a = np.concatenate([base, ties, below, above, np.float32([0.0, -0.0, 1e-30, 3.4e38])])
    np.testing.assert_array_equal(oracle.float_to_bf16(a), _bf16_bits(a))


def test_q8_dequant_bf16_is_rounded_fp32_product():
    rng = np.random.default_rng(7)
    q = rng.integers(-127, 128, size=(16, 64)).astype(np.int8)
    s = (rng.uniform(0.5, 2.0, 16) * 1e-2).astype(np.float32)
    prod = q.astype(np.float32) * s[:, None]            # IEEE fp32 products
    np.testing.assert_array_equal(oracle.dequant_rows(q, s, "bf16"), _bf16_bits(prod))


def test_combine_q8_closed_form():
    """Two kept choices whose payload codes are all 1 with scale s, weights 0.25 and
    0.75: out = x + s exactly; a token with both choices dropped is out = x."""
    N, d, k = 3, 16, 2
    rng = np.random.default_rng(8)
    x = rng.standard_normal((N, d)).astype(np.float32)
    yq = np.ones((4, d), np.int8)
    s = np.float32(0.125)
    yscale = np.full(4, s, np.float32)
    slot_of = np.array([[0, 1], [-1, -1], [3, 2]], np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5], [0.25, 0.75]])
    out = oracle.combine_q8(np.arange(N, dtype=np.int32), x, yq, yscale, slot_of, w)
    np.testing.assert_array_equal(out[0], x[0].astype(np.float64) + 0.125)
    np.testing.assert_array_equal(out[1], x[1].astype(np.float64))
    np.testing.assert_array_equal(out[2], x[2].astype(np.float64) + 0.125)
    # a negative code enters with its sign, weighted by its own choice's weight
    yq[3, :] = -2
    out = oracle.combine_q8(np.arange(N, dtype=np.int32), x, yq, yscale, slot_of, w)
    np.testing.assert_array_equal(out[2], x[2].astype(np.float64) + 0.75 * 0.125 - 0.25 * 0.25)
