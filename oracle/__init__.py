"""CPU oracle for the MoE layer hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg
of ``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never loads it, and it shares no code with them.

This module only marshals numpy arrays into ``libmoe_oracle.so`` (plain C++, see
``moe_oracle.cpp`` for the arithmetic and the passages each step follows).
Activations of dtype bf16 travel as raw ``uint16`` bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

ACT_F32 = 0
ACT_BF16 = 1


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        F = ctypes.c_float
        lib.oracle_sigmoid_spec.restype = F
        lib.oracle_sigmoid_spec.argtypes = [F]
        lib.oracle_sigmoid_spec_many.argtypes = [ctypes.c_int64, P, P]
        lib.oracle_num_threads.restype = I
        lib.oracle_rank_of.argtypes = [I, I, I, I]
        lib.oracle_capacity.argtypes = [I, I, I, F]
        lib.oracle_router_logits.argtypes = [I, I, I, I, P, P, P, P]
        lib.oracle_route.argtypes = [I, I, I, I, I, I, I, P, P, P, P]
        lib.oracle_dispatch.argtypes = [I, I, I, I, I, F, P, P, P, P, P, P, P, P, P]
        lib.oracle_dispatch_mode.argtypes = [I, I, I, I, I, F, I, P, P, P, P, P, P, P, P, P]
        lib.oracle_expert_rows.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P]
        lib.oracle_combine.argtypes = [I, P, I, I, I, P, P, P, P, P, P]
        lib.oracle_layer_tokens.argtypes = [I, P, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P]
        lib.oracle_bias_update.argtypes = [I, I, I, P, F, P]
        lib.oracle_quant_rows.argtypes = [I, I, I, P, P, P, P]
        lib.oracle_dequant_rows.argtypes = [I, I, I, P, P, P, P]
        lib.oracle_combine_q8.argtypes = [I, P, I, I, I, P, P, P, P, P, P, P]
        lib.oracle_float_to_bf16.argtypes = [ctypes.c_int64, P, P]
        lib.oracle_combine_backward.argtypes = [I, I, I, I, P, P, P, P, P, P]
        lib.oracle_ffn_backward_rows.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, P]
        lib.oracle_ffn_wgrad.argtypes = [I, I, I, I, P, P, P, P, I, P, P, P, P]
        lib.oracle_route_backward.argtypes = [I, I, I, I, I, P, P, P, P]
        lib.oracle_router_grads.argtypes = [I, I, I, I, P, P, P, I, P, P, P, P]
        lib.oracle_dispatch_backward.argtypes = [I, P, I, I, I, P, P, P, P, P, P]
        _LIB = lib
    return _LIB


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _act(a):
    """Return (contiguous array, act_dtype code) for fp32 or bf16-bits arrays."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, ACT_F32
    if a.dtype == np.uint16:
        return a, ACT_BF16
    raise TypeError(f"activation arrays must be float32 or uint16 (bf16 bits), got {a.dtype}")


def _tokens(tokens, N):
    """Token indices as int32, every one a row of the N-token batch (the C side reads
    row t of x, slot_of and the weights without a bounds check)."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
    if tokens.size and (tokens.min() < 0 or tokens.max() >= N):
        raise ValueError(f"token index outside the batch of {N} tokens")
    return tokens


def num_threads():
    return _lib().oracle_num_threads()


def sigmoid_spec(l):
    l = np.ascontiguousarray(l, dtype=np.float32)
    out = np.empty_like(l)
    _lib().oracle_sigmoid_spec_many(l.size, _p(l), _p(out))
    return out


def rank_of(e, E, R, rank_map):
    return _lib().oracle_rank_of(e, E, R, rank_map)


def capacity(N, k, E, cf):
    return _lib().oracle_capacity(N, k, E, float(cf))


def router_logits(x, w, b=None):
    x, code = _act(x)
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, d = x.shape
    E = w.shape[0]
    bb = None if b is None else np.ascontiguousarray(b, dtype=np.float32)
    out = np.empty((N, E), dtype=np.float32)
    rc = _lib().oracle_router_logits(N, d, E, code, _p(x), _p(w), _p(bb), _p(out))
    assert rc == 0
    return out


def route(logits, k, score_fn=0, normalize=True, num_groups=1, topk_groups=1, sel_bias=None):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    N, E = logits.shape
    sb = None if sel_bias is None else np.ascontiguousarray(sel_bias, dtype=np.float32)
    idx = np.empty((N, k), dtype=np.int32)
    w = np.empty((N, k), dtype=np.float64)
    rc = _lib().oracle_route(N, E, k, score_fn, int(bool(normalize)), num_groups, topk_groups,
                             _p(logits), _p(sb), _p(idx), _p(w))
    if rc != 0:
        raise ValueError(f"oracle_route rejected the arguments (rc={rc})")
    return idx, w


def dispatch(idx, E, R, rank_map=0, cf=0.0, mode=0):
    """Counting, capacity and send order.  mode 0: packed, token-order priority;
    mode 1: capacity-padded [E, C] slots, choice-major priority (needs cf > 0)."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    N, k = idx.shape
    A = N * k
    C = capacity(N, k, E, cf)
    rows = A if mode == 0 else E * C
    out = dict(
        expert_counts=np.empty(E, np.int32), kept_counts=np.empty(E, np.int32),
        expert_start=np.empty(E, np.int32), rank_counts=np.empty(R, np.int32),
        rank_offsets=np.empty(R + 1, np.int32), slot_of=np.empty(A, np.int32),
        perm_src=np.empty(max(rows, 1), np.int32), num_kept=np.empty(1, np.int32))
    rc = _lib().oracle_dispatch_mode(N, E, k, R, rank_map, float(cf), int(mode), _p(idx),
                                     *[_p(out[n]) for n in ("expert_counts", "kept_counts",
                                                            "expert_start", "rank_counts",
                                                            "rank_offsets", "slot_of", "perm_src",
                                                            "num_kept")])
    if rc != 0:
        raise ValueError(f"oracle_dispatch rejected the arguments (rc={rc})")
    out["perm_src"] = out["perm_src"][:rows]
    out["num_kept"] = int(out["num_kept"][0])
    out["capacity"] = C
    out["send_rows"] = rows
    return out


def expert_rows(xrows, expert, w_gate_up, w_down, shared_gate_up=None, shared_down=None):
    """y[i] = FFN_{expert[i]}(xrows[i]) in fp64; expert id E selects the shared expert."""
    xrows, code = _act(xrows)
    wgu, c2 = _act(w_gate_up)
    wd, c3 = _act(w_down)
    assert code == c2 == c3
    n, d = xrows.shape
    E, twoF, _ = wgu.shape
    F = twoF // 2
    sgu = sd = None
    Fs = 0
    if shared_gate_up is not None:
        sgu, _ = _act(shared_gate_up)
        sd, _ = _act(shared_down)
        Fs = sgu.shape[0] // 2
    expert = np.ascontiguousarray(expert, dtype=np.int32)
    y = np.empty((n, d), dtype=np.float64)
    _lib().oracle_expert_rows(n, d, E, F, Fs, code, _p(xrows), _p(expert), _p(wgu), _p(wd),
                              _p(sgu), _p(sd), _p(y))
    return y


def combine(tokens, x, yperm, slot_of, w, ys=None):
    x, code = _act(x)
    yperm, c2 = _act(yperm)
    assert code == c2
    N, d = x.shape
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32).reshape(-1)
    w = np.ascontiguousarray(w, dtype=np.float64).reshape(-1)
    k = slot_of.size // N
    if ys is not None:
        ys, c3 = _act(ys)
        assert c3 == code
    tokens = _tokens(tokens, N)
    out = np.empty((tokens.size, d), dtype=np.float64)
    _lib().oracle_combine(tokens.size, _p(tokens), d, k, code, _p(x), _p(yperm), _p(ys),
                          _p(slot_of), _p(w), _p(out))
    return out


def layer_tokens(tokens, x, idx, w, slot_of, w_gate_up, w_down, shared_gate_up=None,
                 shared_down=None):
    """Full layer output (fp64) for the listed tokens, routing given."""
    x, code = _act(x)
    wgu, _ = _act(w_gate_up)
    wd, _ = _act(w_down)
    N, d = x.shape
    E, twoF, _ = wgu.shape
    F = twoF // 2
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    k = idx.shape[1]
    w = np.ascontiguousarray(w, dtype=np.float64)
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32).reshape(-1)
    sgu = sd = None
    Fs = 0
    if shared_gate_up is not None:
        sgu, _ = _act(shared_gate_up)
        sd, _ = _act(shared_down)
        Fs = sgu.shape[0] // 2
    tokens = _tokens(tokens, N)
    out = np.empty((tokens.size, d), dtype=np.float64)
    _lib().oracle_layer_tokens(tokens.size, _p(tokens), d, E, k, F, Fs, code, _p(x), _p(idx),
                               _p(w), _p(slot_of), _p(wgu), _p(wd), _p(sgu), _p(sd), _p(out))
    return out


def bias_update(counts, bias, N, k, step):
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    b = np.array(bias, dtype=np.float32, copy=True)
    _lib().oracle_bias_update(b.size, N, k, _p(counts), float(step), _p(b))
    return b


def quant_rows(rows, valid=None):
    """Per-row symmetric INT8 codes and fp32 scales of rows [R, d] (fp32 or bf16 bits).
    Rows with valid[r] < 0 are skipped (codes 0, scale NaN in the returned arrays)."""
    rows, code = _act(rows)
    R, d = rows.shape
    q = np.zeros((R, d), np.int8)
    s = np.full(R, np.nan, np.float32)
    v = None if valid is None else np.ascontiguousarray(valid, dtype=np.int32)
    _lib().oracle_quant_rows(R, d, code, _p(rows), _p(v), _p(q), _p(s))
    return q, s


def dequant_rows(q, scale, act_dtype="bf16", valid=None):
    """(float)q * scale per row, stored as fp32 or bf16 bits (uint16)."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    R, d = q.shape
    code = ACT_F32 if act_dtype == "f32" else ACT_BF16
    out = np.zeros((R, d), np.float32 if code == ACT_F32 else np.uint16)
    v = None if valid is None else np.ascontiguousarray(valid, dtype=np.int32)
    _lib().oracle_dequant_rows(R, d, code, _p(q), _p(scale), _p(v), _p(out))
    return out


def combine_q8(tokens, x, yq, yscale, slot_of, w, ys=None):
    x, code = _act(x)
    N, d = x.shape
    yq = np.ascontiguousarray(yq, dtype=np.int8)
    yscale = np.ascontiguousarray(yscale, dtype=np.float32)
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32).reshape(-1)
    w = np.ascontiguousarray(w, dtype=np.float64).reshape(-1)
    k = slot_of.size // N
    if ys is not None:
        ys, c3 = _act(ys)
        assert c3 == code
    tokens = _tokens(tokens, N)
    out = np.empty((tokens.size, d), dtype=np.float64)
    _lib().oracle_combine_q8(tokens.size, _p(tokens), d, k, code, _p(x), _p(yq), _p(yscale),
                             _p(ys), _p(slot_of), _p(w), _p(out))
    return out


def float_to_bf16(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    _lib().oracle_float_to_bf16(a.size, _p(a), _p(out))
    return out


# ------------------------------------------------------------------ backward

def combine_backward(dout, yperm, slot_of, w):
    """dy [S, d] fp64 (written at kept slots, 0 elsewhere) and dw [N, k] fp64."""
    dout, code = _act(dout)
    yperm, c2 = _act(yperm)
    assert code == c2
    N, d = dout.shape
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32).reshape(-1)
    k = slot_of.size // N
    w = np.ascontiguousarray(w, dtype=np.float64).reshape(-1)
    dy = np.zeros((yperm.shape[0], d), np.float64)
    dw = np.empty(N * k, np.float64)
    _lib().oracle_combine_backward(N, d, k, code, _p(dout), _p(yperm), _p(slot_of), _p(w),
                                   _p(dy), _p(dw))
    return dy, dw.reshape(N, k)


def ffn_backward_rows(xrows, dyrows, expert, w_gate_up, w_down, shared_gate_up=None,
                      shared_down=None):
    """dx [n, d] fp64 of each row through its expert (expert id E = the shared expert)."""
    xrows, code = _act(xrows)
    dyrows, c1 = _act(dyrows)
    assert code == c1
    wgu, _ = _act(w_gate_up)
    wd, _ = _act(w_down)
    n, d = xrows.shape
    E, twoF, _ = wgu.shape
    sgu = sd = None
    Fs = 0
    if shared_gate_up is not None:
        sgu, _ = _act(shared_gate_up)
        sd, _ = _act(shared_down)
        Fs = sgu.shape[0] // 2
    expert = np.ascontiguousarray(expert, dtype=np.int32)
    dx = np.empty((n, d), np.float64)
    _lib().oracle_ffn_backward_rows(n, d, E, twoF // 2, Fs, code, _p(xrows), _p(dyrows),
                                    _p(expert), _p(wgu), _p(wd), _p(sgu), _p(sd), _p(dx))
    return dx


def ffn_wgrad(xrows, dyrows, wgu_e, wd_e, fs=None):
    """Weight gradients of one expert from its rows: for each hidden unit f in fs
    (default all), dWd[:, f], dWg[f, :], dWu[f, :] as three [nf, d] fp64 arrays."""
    xrows, code = _act(xrows)
    dyrows, c1 = _act(dyrows)
    assert code == c1
    wgu_e, _ = _act(wgu_e)
    wd_e, _ = _act(wd_e)
    n, d = xrows.shape
    Fx = wgu_e.shape[0] // 2
    fs = np.arange(Fx, dtype=np.int32) if fs is None else np.ascontiguousarray(fs, np.int32)
    nf = fs.size
    out = [np.empty((nf, d), np.float64) for _ in range(3)]
    _lib().oracle_ffn_wgrad(n, d, Fx, code, _p(xrows), _p(dyrows), _p(wgu_e), _p(wd_e), nf, _p(fs),
                            *[_p(o) for o in out])
    return out


def route_backward(logits, idx, dw, score_fn=0, normalize=True):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    N, E = logits.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    k = idx.shape[1]
    dw = np.ascontiguousarray(dw, dtype=np.float64)
    dl = np.empty((N, E), np.float64)
    _lib().oracle_route_backward(N, E, k, score_fn, int(bool(normalize)), _p(logits), _p(idx),
                                 _p(dw), _p(dl))
    return dl


def router_grads(x, w_router, dl, tokens=None, params=True):
    """(dx_router [ntok, d], dWr [E, d] or None, db [E] or None), fp64."""
    x, code = _act(x)
    N, d = x.shape
    Wr = np.ascontiguousarray(w_router, dtype=np.float32)
    E = Wr.shape[0]
    dl = np.ascontiguousarray(dl, dtype=np.float64)
    tokens = np.arange(N, dtype=np.int32) if tokens is None else \
        np.ascontiguousarray(tokens, dtype=np.int32)
    dxr = np.empty((tokens.size, d), np.float64)
    dwr = np.empty((E, d), np.float64) if params else None
    db = np.empty(E, np.float64) if params else None
    _lib().oracle_router_grads(N, d, E, code, _p(x), _p(Wr), _p(dl), tokens.size, _p(tokens),
                               _p(dxr), _p(dwr), _p(db))
    return dxr, dwr, db


def dispatch_backward(tokens, dout, dxperm, slot_of, dxs=None, dxr=None):
    dout, code = _act(dout)
    dxperm, c1 = _act(dxperm)
    assert code == c1
    N, d = dout.shape
    slot_of = np.ascontiguousarray(slot_of, dtype=np.int32).reshape(-1)
    k = slot_of.size // N
    if dxs is not None:
        dxs, c2 = _act(dxs)
        assert c2 == code
    dxr = None if dxr is None else np.ascontiguousarray(dxr, dtype=np.float32)
    tokens = _tokens(tokens, N)
    out = np.empty((tokens.size, d), np.float64)
    _lib().oracle_dispatch_backward(tokens.size, _p(tokens), d, k, code, _p(dout), _p(dxs),
                                    _p(dxr), _p(dxperm), _p(slot_of), _p(out))
    return out
