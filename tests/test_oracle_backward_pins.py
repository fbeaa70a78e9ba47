"""Pins of the oracle's backward pass (CPU only).

The gradients the oracle derives by hand are checked against
  * central finite differences of the oracle's own forward layer (which is pinned by
    test_oracle_pins.py), Richardson-extrapolated, on tiny layers of every routing
    variant: a sign slip, a dropped term, a transposed weight or a wrong router
    Jacobian fails them;
  * torch autograd on the dense special case (one expert, top-1), a library routine;
  * closed forms: a token whose every choice was dropped passes dout through unchanged.
Loss L = sum(G * out) with a fixed random G, so dL/dout = G.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle

F32 = np.float32


@dataclasses.dataclass
class Tiny:
    x: np.ndarray
    Wr: np.ndarray
    b: np.ndarray
    sel: np.ndarray
    wgu: np.ndarray
    wd: np.ndarray
    sgu: np.ndarray
    sd: np.ndarray
    G: np.ndarray
    k: int
    score_fn: int
    normalize: bool
    groups: int
    topk_groups: int
    cf: float


def make(seed, N=7, d=8, E=4, k=2, F=4, Fs=4, score_fn=1, normalize=True, groups=2,
         topk_groups=1, cf=0.0):
    rng = np.random.default_rng(seed)
    r = lambda *s, sc=1.0: (rng.standard_normal(s) * sc).astype(F32)
    return Tiny(x=r(N, d), Wr=r(E, d, sc=0.6), b=r(E, sc=0.2),
                sel=r(E, sc=0.05) if score_fn == 1 else None,
                wgu=r(E, 2 * F, d, sc=0.4), wd=r(E, d, F, sc=0.4),
                sgu=r(2 * Fs, d, sc=0.4) if Fs else None, sd=r(d, Fs, sc=0.4) if Fs else None,
                G=r(N, d), k=k, score_fn=score_fn, normalize=normalize, groups=groups,
                topk_groups=topk_groups, cf=cf)


def forward(P):
    N = P.x.shape[0]
    E = P.Wr.shape[0]
    logits = oracle.router_logits(P.x, P.Wr, P.b)
    idx, w = oracle.route(logits, P.k, P.score_fn, P.normalize, P.groups, P.topk_groups, P.sel)
    dd = oracle.dispatch(idx, E, min(2, E), 0, P.cf)
    out = oracle.layer_tokens(np.arange(N, dtype=np.int32), P.x, idx, w, dd["slot_of"], P.wgu,
                              P.wd, P.sgu, P.sd)
    return float((P.G.astype(np.float64) * out).sum()), idx, dd["slot_of"]


def backward(P):
    """Every gradient through the oracle's backward functions."""
    N, d = P.x.shape
    E, k = P.Wr.shape[0], P.k
    logits = oracle.router_logits(P.x, P.Wr, P.b)
    idx, w = oracle.route(logits, k, P.score_fn, P.normalize, P.groups, P.topk_groups, P.sel)
    dd = oracle.dispatch(idx, E, min(2, E), 0, P.cf)
    ps = dd["perm_src"]
    kept = np.nonzero(ps >= 0)[0]
    tok, exp = ps[kept] // k, idx.reshape(-1)[ps[kept]]
    S = dd["send_rows"]
    yperm = np.zeros((S, d), F32)
    yperm[kept] = oracle.expert_rows(P.x[tok], exp, P.wgu, P.wd).astype(F32)
    dy, dw = oracle.combine_backward(P.G, yperm, dd["slot_of"], w)
    dxperm = np.zeros((S, d), F32)
    if kept.size:
        dxperm[kept] = oracle.ffn_backward_rows(P.x[tok], dy[kept].astype(F32), exp, P.wgu,
                                                P.wd).astype(F32)
    dxs = None
    if P.sgu is not None:
        dxs = oracle.ffn_backward_rows(P.x, P.G, np.full(N, E, np.int32), P.wgu, P.wd, P.sgu,
                                       P.sd).astype(F32)
    dl = oracle.route_backward(logits, idx, dw, P.score_fn, P.normalize)
    dxr, dWr, db = oracle.router_grads(P.x, P.Wr, dl)
    dx = oracle.dispatch_backward(np.arange(N, dtype=np.int32), P.G, dxperm, dd["slot_of"], dxs,
                                  dxr.astype(F32))
    dwgu = np.zeros(P.wgu.shape)
    dwd = np.zeros(P.wd.shape)
    for e in range(E):
        s0, n = dd["expert_start"][e], dd["kept_counts"][e]
        if n == 0:
            continue
        rows = np.arange(s0, s0 + n)
        cd, rg, ru = oracle.ffn_wgrad(P.x[ps[rows] // k], dy[rows].astype(F32), P.wgu[e], P.wd[e])
        dwd[e] = cd.T
        dwgu[e] = np.vstack([rg, ru])
    g = dict(x=dx, Wr=dWr, b=db, wgu=dwgu, wd=dwd, dw=dw, dl=dl, slot_of=dd["slot_of"])
    if P.sgu is not None:
        cd, rg, ru = oracle.ffn_wgrad(P.x, P.G, P.sgu, P.sd)
        g["sd"] = cd.T
        g["sgu"] = np.vstack([rg, ru])
    return g


def fd(P, name, index):
    """Richardson-extrapolated central difference of L in P.<name>[index] (the step
    actually taken is the fp32-representable one); None if the selection moved."""
    arr = getattr(P, name)
    v0 = arr[index]
    L0, idx0, slot0 = forward(P)
    ds = []
    for h in (2.0 ** -7, 2.0 ** -8):
        vals = []
        steps = []
        for sgn in (1, -1):
            v = F32(float(v0) + sgn * h)
            arr[index] = v
            L, idx, slot = forward(P)
            arr[index] = v0
            if not (np.array_equal(idx, idx0) and np.array_equal(slot, slot0)):
                return None
            vals.append(L)
            steps.append(float(v))
        ds.append((vals[0] - vals[1]) / (steps[0] - steps[1]))
    return (4 * ds[1] - ds[0]) / 3


VARIANTS = {
    "sigmoid_norm_groups_shared": dict(score_fn=1, normalize=True, groups=2, topk_groups=1),
    "sigmoid_unnorm": dict(score_fn=1, normalize=False, groups=1, topk_groups=1, Fs=0),
    "softmax_norm_capacity": dict(score_fn=0, normalize=True, groups=1, topk_groups=1, Fs=0,
                                  cf=0.6),
    "softmax_unnorm_shared": dict(score_fn=0, normalize=False, groups=1, topk_groups=1),
}


@pytest.mark.parametrize("name", list(VARIANTS))
def test_backward_matches_finite_differences(name):
    P = make(11, **VARIANTS[name])
    g = backward(P)
    rng = np.random.default_rng(3)
    params = ["x", "Wr", "b", "wgu", "wd"] + (["sgu", "sd"] if P.sgu is not None else [])
    checked = 0
    for p in params:
        arr = getattr(P, p)
        scale = np.max(np.abs(g[p])) + 1e-12
        picks = [tuple(rng.integers(0, s) for s in arr.shape) for _ in range(6)]
        if p == "wgu":   # a gate row and an up row of an expert that has kept rows
            e = int(np.argmax([np.any(g["wgu"][i]) for i in range(arr.shape[0])]))
            F = arr.shape[1] // 2
            picks += [(e, 1, 2), (e, F + 1, 2)]
        for ix in picks:
            num = fd(P, p, ix)
            if num is None:
                continue
            assert abs(num - g[p][ix]) <= 1e-3 * scale, (p, ix, num, g[p][ix])
            checked += 1
    assert checked >= 20


def test_softmax_capacity_case_drops_something():
    """The capacity variant above really has dropped choices (so the dw = 0 path and
    the router Jacobian of a partly dropped token are exercised)."""
    P = make(11, **VARIANTS["softmax_norm_capacity"])
    g = backward(P)
    assert np.any(g["slot_of"] < 0)
    dropped = g["slot_of"].reshape(P.x.shape[0], P.k) < 0
    assert np.all(g["dw"][dropped] == 0.0)


def test_fully_dropped_token_passes_dout_through():
    """No shared expert; a token whose every choice was dropped: its dw are 0, so its
    logit gradient is 0 (normalised routing) and dx = dout exactly."""
    P = make(5, N=9, score_fn=0, normalize=True, groups=1, topk_groups=1, Fs=0, cf=0.25)
    g = backward(P)
    slot = g["slot_of"].reshape(9, P.k)
    full = np.nonzero((slot < 0).all(1))[0]
    assert full.size > 0
    assert np.all(g["dl"][full] == 0.0)
    np.testing.assert_array_equal(g["x"][full], P.G[full].astype(np.float64))


def test_dense_single_expert_matches_torch_autograd():
    """E = 1, k = 1, normalised softmax: weight 1 and no router gradient; the layer is
    x + SwiGLU(x) (+ shared), whose gradients torch autograd computes in fp64."""
    P = make(7, N=5, d=12, E=1, k=1, F=6, Fs=5, score_fn=0, normalize=True, groups=1,
             topk_groups=1)
    g = backward(P)
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    x, wgu, wd, sgu, sd = t(P.x), t(P.wgu[0]), t(P.wd[0]), t(P.sgu), t(P.sd)

    def swiglu(z, wgu_, wd_):
        F = wgu_.shape[0] // 2
        gu = z @ wgu_.T
        return (torch.nn.functional.silu(gu[:, :F]) * gu[:, F:]) @ wd_.T

    out = x + swiglu(x, wgu, wd) + swiglu(x, sgu, sd)
    (torch.tensor(P.G, dtype=torch.float64) * out).sum().backward()
    for name, ref, got in (("x", x.grad, g["x"]), ("wgu", wgu.grad, g["wgu"][0]),
                           ("wd", wd.grad, g["wd"][0]), ("sgu", sgu.grad, g["sgu"]),
                           ("sd", sd.grad, g["sd"])):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-6, atol=1e-6, err_msg=name)
    assert np.all(g["dl"] == 0.0) and np.all(g["Wr"] == 0.0)
