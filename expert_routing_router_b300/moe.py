"""ctypes binding of libmoe.so -- argument marshalling only.

Every function below has the name of the C entry point it calls (include/moe.h)
and forwards torch tensors as raw device pointers.  No step of the layer runs in
Python: if the library is missing the import-time loader raises, and there is no
fallback of any kind.  Tensors must already be on the GPU with the layouts the
header documents.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA = range(5)
DTYPE_F32, DTYPE_BF16 = 0, 1


class moe_config(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("num_ranks", ctypes.c_int32), ("rank_map", ctypes.c_int32),
                ("score_fn", ctypes.c_int32), ("normalize_topk", ctypes.c_int32),
                ("num_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("d_ff", ctypes.c_int32),
                ("shared_d_ff", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
                ("dispatch_mode", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)}")


EXPORTS = ("moe_send_rows", "moe_workspace_size", "moe_route", "moe_dispatch", "moe_dispatch_noalloc",
           "moe_expert_ffn", "moe_selftest_ffn_stall", "moe_combine", "moe_bias_update",
           "moe_dispatch_q8", "moe_quant_rows", "moe_dequant_rows", "moe_combine_q8",
           "moe_backward_workspace_size", "moe_combine_backward", "moe_expert_ffn_backward",
           "moe_saved_size", "moe_expert_ffn_save",
           "moe_route_backward", "moe_dispatch_backward", "moe_status_string")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe.so is not built ({LIB_PATH}); run "
                          "`python expert_routing_router_b300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    P, S, I, F = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    C = ctypes.POINTER(moe_config)
    lib.moe_workspace_size.argtypes = [C, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_send_rows.argtypes = [C, ctypes.POINTER(ctypes.c_int64)]
    lib.moe_route.argtypes = [C] + [P] * 8 + [S, P]
    lib.moe_dispatch.argtypes = [C] + [P] * 12 + [S, P]
    lib.moe_dispatch_noalloc.argtypes = [C] + [P] * 11 + [P]
    lib.moe_expert_ffn.argtypes = [C] + [P] * 11 + [S, P]
    lib.moe_selftest_ffn_stall.argtypes = [C] + [P] * 11 + [S, P]
    lib.moe_combine.argtypes = [C] + [P] * 6 + [P]
    lib.moe_bias_update.argtypes = [C, P, P, F, P]
    lib.moe_dispatch_q8.argtypes = [C] + [P] * 13 + [S, P]
    lib.moe_quant_rows.argtypes = [C] + [P] * 4 + [P]
    lib.moe_dequant_rows.argtypes = [C] + [P] * 4 + [P]
    lib.moe_combine_q8.argtypes = [C] + [P] * 7 + [P]
    lib.moe_backward_workspace_size.argtypes = [C, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_combine_backward.argtypes = [C] + [P] * 6 + [P]
    lib.moe_expert_ffn_backward.argtypes = [C] + [P] * 18 + [S, P]
    lib.moe_saved_size.argtypes = [C, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_expert_ffn_save.argtypes = [C] + [P] * 11 + [S, P, S, P]
    lib.moe_route_backward.argtypes = [C] + [P] * 9 + [P, S, P]
    lib.moe_dispatch_backward.argtypes = [C] + [P] * 6 + [P]
    lib.moe_status_string.argtypes = [I]
    lib.moe_status_string.restype = ctypes.c_char_p
    for fn in EXPORTS[:-1]:
        getattr(lib, fn).restype = I
    return lib


_lib = _load()
lib = _lib


def status_string(status):
    return _lib.moe_status_string(int(status)).decode()


def config(w):
    """moe_config for a workloads.Workload (or any object with the same fields)."""
    return moe_config(w.tokens, w.hidden, w.num_experts, w.top_k, w.num_ranks, w.rank_map,
                      w.score_fn, int(bool(w.normalize_topk)), w.num_groups, w.topk_groups,
                      float(w.capacity_factor), w.d_ff, w.shared_d_ff,
                      DTYPE_F32 if w.act_dtype == "f32" else DTYPE_BF16,
                      int(getattr(w, "dispatch_mode", 0)))


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, status):
    if status != MOE_OK:
        raise MoeError(fn, status)


def moe_send_rows(cfg):
    n = ctypes.c_int64(0)
    _check("moe_send_rows", _lib.moe_send_rows(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def moe_workspace_size(cfg):
    n = ctypes.c_size_t(0)
    _check("moe_workspace_size", _lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def moe_route(cfg, x, w_router, b_router, sel_bias, logits, topk_idx, topk_w, workspace,
              stream=None):
    _check("moe_route", _lib.moe_route(
        ctypes.byref(cfg), _p(x), _p(w_router), _p(b_router), _p(sel_bias), _p(logits),
        _p(topk_idx), _p(topk_w), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def moe_dispatch(cfg, topk_idx, x, xperm, expert_counts, kept_counts, expert_start, rank_counts,
                 rank_offsets, slot_of, perm_src, num_kept, workspace, stream=None):
    _check("moe_dispatch", _lib.moe_dispatch(
        ctypes.byref(cfg), _p(topk_idx), _p(x), _p(xperm), _p(expert_counts), _p(kept_counts),
        _p(expert_start), _p(rank_counts), _p(rank_offsets), _p(slot_of), _p(perm_src),
        _p(num_kept), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def moe_dispatch_noalloc(cfg, topk_idx, x, xperm, expert_counts, kept_counts, expert_start,
                         rank_counts, rank_offsets, slot_of, perm_src, num_kept, stream=None):
    """moe_dispatch for callers that cannot allocate: no workspace argument; the scratch
    is a static array inside the library (see include/moe.h for limits and caveats)."""
    _check("moe_dispatch_noalloc", _lib.moe_dispatch_noalloc(
        ctypes.byref(cfg), _p(topk_idx), _p(x), _p(xperm), _p(expert_counts), _p(kept_counts),
        _p(expert_start), _p(rank_counts), _p(rank_offsets), _p(slot_of), _p(perm_src),
        _p(num_kept), _stream(stream)))


def moe_expert_ffn(cfg, xperm, expert_start, kept_counts, w_gate_up, w_down, x, shared_gate_up,
                   shared_down, yperm, yshared, workspace, stream=None):
    _check("moe_expert_ffn", _lib.moe_expert_ffn(
        ctypes.byref(cfg), _p(xperm), _p(expert_start), _p(kept_counts), _p(w_gate_up),
        _p(w_down), _p(x), _p(shared_gate_up), _p(shared_down), _p(yperm), _p(yshared),
        _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_selftest_ffn_stall(cfg, xperm, expert_start, kept_counts, w_gate_up, w_down, x,
                           shared_gate_up, shared_down, yperm, yshared, workspace, stream=None):
    """Failure-handling self-test: the prefill expert kernels with one pipeline slot never
    loaded (outputs invalid; the workspace status word becomes nonzero)."""
    _check("moe_selftest_ffn_stall", _lib.moe_selftest_ffn_stall(
        ctypes.byref(cfg), _p(xperm), _p(expert_start), _p(kept_counts), _p(w_gate_up),
        _p(w_down), _p(x), _p(shared_gate_up), _p(shared_down), _p(yperm), _p(yshared),
        _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_combine(cfg, yperm, slot_of, topk_w, residual, yshared, out, stream=None):
    _check("moe_combine", _lib.moe_combine(
        ctypes.byref(cfg), _p(yperm), _p(slot_of), _p(topk_w), _p(residual), _p(yshared),
        _p(out), _stream(stream)))


def moe_bias_update(cfg, expert_counts, sel_bias, step, stream=None):
    _check("moe_bias_update", _lib.moe_bias_update(
        ctypes.byref(cfg), _p(expert_counts), _p(sel_bias), float(step), _stream(stream)))


def moe_dispatch_q8(cfg, topk_idx, x, xperm_q, xscale, expert_counts, kept_counts, expert_start,
                    rank_counts, rank_offsets, slot_of, perm_src, num_kept, workspace, stream=None):
    _check("moe_dispatch_q8", _lib.moe_dispatch_q8(
        ctypes.byref(cfg), _p(topk_idx), _p(x), _p(xperm_q), _p(xscale), _p(expert_counts),
        _p(kept_counts), _p(expert_start), _p(rank_counts), _p(rank_offsets), _p(slot_of),
        _p(perm_src), _p(num_kept), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def moe_quant_rows(cfg, rows, perm_src, q, scale, stream=None):
    _check("moe_quant_rows", _lib.moe_quant_rows(
        ctypes.byref(cfg), _p(rows), _p(perm_src), _p(q), _p(scale), _stream(stream)))


def moe_dequant_rows(cfg, q, scale, perm_src, rows, stream=None):
    _check("moe_dequant_rows", _lib.moe_dequant_rows(
        ctypes.byref(cfg), _p(q), _p(scale), _p(perm_src), _p(rows), _stream(stream)))


def moe_combine_q8(cfg, yperm_q, yscale, slot_of, topk_w, residual, yshared, out, stream=None):
    _check("moe_combine_q8", _lib.moe_combine_q8(
        ctypes.byref(cfg), _p(yperm_q), _p(yscale), _p(slot_of), _p(topk_w), _p(residual),
        _p(yshared), _p(out), _stream(stream)))


# ------------------------------------------------------------------ backward

def moe_backward_workspace_size(cfg):
    n = ctypes.c_size_t(0)
    _check("moe_backward_workspace_size",
           _lib.moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def moe_combine_backward(cfg, dout, yperm, slot_of, topk_w, dyperm, dtopk_w, stream=None):
    _check("moe_combine_backward", _lib.moe_combine_backward(
        ctypes.byref(cfg), _p(dout), _p(yperm), _p(slot_of), _p(topk_w), _p(dyperm),
        _p(dtopk_w), _stream(stream)))


def moe_expert_ffn_backward(cfg, xperm, expert_start, kept_counts, w_gate_up, w_down, x,
                            shared_gate_up, shared_down, dyperm, dout, dxperm, dx_shared,
                            dw_gate_up, dw_down, dshared_gate_up, dshared_down, workspace,
                            stream=None, saved=None):
    _check("moe_expert_ffn_backward", _lib.moe_expert_ffn_backward(
        ctypes.byref(cfg), _p(xperm), _p(expert_start), _p(kept_counts), _p(w_gate_up),
        _p(w_down), _p(x), _p(shared_gate_up), _p(shared_down), _p(dyperm), _p(dout),
        _p(dxperm), _p(dx_shared), _p(dw_gate_up), _p(dw_down), _p(dshared_gate_up),
        _p(dshared_down), _p(saved), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_saved_size(cfg):
    n = ctypes.c_size_t(0)
    _check("moe_saved_size", _lib.moe_saved_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def moe_expert_ffn_save(cfg, xperm, expert_start, kept_counts, w_gate_up, w_down, x,
                        shared_gate_up, shared_down, yperm, yshared, saved, workspace,
                        stream=None):
    """moe_expert_ffn that also keeps h and g|u in `saved` for the backward pass."""
    _check("moe_expert_ffn_save", _lib.moe_expert_ffn_save(
        ctypes.byref(cfg), _p(xperm), _p(expert_start), _p(kept_counts), _p(w_gate_up),
        _p(w_down), _p(x), _p(shared_gate_up), _p(shared_down), _p(yperm), _p(yshared),
        _p(saved), saved.numel() * saved.element_size(), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_route_backward(cfg, x, w_router, logits, topk_idx, dtopk_w, dlogits, dx_router,
                       dw_router, db_router, workspace=None, stream=None):
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("moe_route_backward", _lib.moe_route_backward(
        ctypes.byref(cfg), _p(x), _p(w_router), _p(logits), _p(topk_idx), _p(dtopk_w),
        _p(dlogits), _p(dx_router), _p(dw_router), _p(db_router), _p(workspace), nbytes,
        _stream(stream)))


def moe_dispatch_backward(cfg, dxperm, slot_of, dout, dx_shared, dx_router, dx, stream=None):
    _check("moe_dispatch_backward", _lib.moe_dispatch_backward(
        ctypes.byref(cfg), _p(dxperm), _p(slot_of), _p(dout), _p(dx_shared), _p(dx_router),
        _p(dx), _stream(stream)))


class GradBuffers:
    """Device buffers of one backward call (bf16 layers): gradients of the hidden
    states, every weight and the router, plus the intermediates and the workspace."""

    def __init__(self, w, device="cuda"):
        N, d, E, k, F, Fs = w.tokens, w.hidden, w.num_experts, w.top_k, w.d_ff, w.shared_d_ff
        dt = w.torch_dtype
        f32 = dict(dtype=torch.float32, device=device)
        self.cfg = config(w)
        S = moe_send_rows(self.cfg)
        self.dyperm = torch.empty(S, d, dtype=dt, device=device)
        self.dtopk_w = torch.empty(N, k, **f32)
        self.dxperm = torch.empty(S, d, dtype=dt, device=device)
        self.dx_shared = torch.empty(N, d, dtype=dt, device=device) if Fs else None
        self.dlogits = torch.empty(N, E, **f32)
        self.dx_router = torch.empty(N, d, **f32)
        self.dw_router = torch.empty(E, d, **f32)
        self.db_router = torch.empty(E, **f32)
        self.dx = torch.empty(N, d, dtype=dt, device=device)
        self.dw_gate_up = torch.empty(E, 2 * F, d, dtype=dt, device=device)
        self.dw_down = torch.empty(E, d, F, dtype=dt, device=device)
        self.dshared_gate_up = torch.empty(2 * Fs, d, dtype=dt, device=device) if Fs else None
        self.dshared_down = torch.empty(d, Fs, dtype=dt, device=device) if Fs else None
        self.workspace = torch.empty(moe_backward_workspace_size(self.cfg), dtype=torch.uint8,
                                     device=device)
        self.workspace[:256].zero_()          # sticky device status word starts at 0


def run_layer_backward(b, g, inp, dout, stream=None, saved=None):
    """Backward of the layer pass held in LayerBuffers b (selection fixed), from dout:
    combine, expert FFN (dgrad, wgrad; g, u and h from `saved` if the forward kept them
    with moe_expert_ffn_save, else recomputed), router, dispatch.  Writes every gradient
    into GradBuffers g and returns g.dx."""
    c = b.cfg
    moe_combine_backward(c, dout, b.yperm, b.slot_of, b.topk_w, g.dyperm, g.dtopk_w, stream)
    moe_expert_ffn_backward(c, b.xperm, b.expert_start, b.kept_counts, inp["w_gate_up"],
                            inp["w_down"], inp["x"], inp["shared_gate_up"], inp["shared_down"],
                            g.dyperm, dout, g.dxperm, g.dx_shared, g.dw_gate_up, g.dw_down,
                            g.dshared_gate_up, g.dshared_down, g.workspace, stream, saved)
    moe_route_backward(c, inp["x"], inp["w_router"], b.logits, b.topk_idx, g.dtopk_w, g.dlogits,
                       g.dx_router, g.dw_router, g.db_router, g.workspace, stream)
    moe_dispatch_backward(c, g.dxperm, b.slot_of, dout, g.dx_shared, g.dx_router, g.dx, stream)
    return g.dx


class LayerBuffers:
    """Device buffers of one layer call, sized for the worst case (every assignment
    kept; the capacity-padded layout has E*C send rows)."""

    def __init__(self, w, device="cuda"):
        N, d, E, k, R = w.tokens, w.hidden, w.num_experts, w.top_k, w.num_ranks
        dt = w.torch_dtype
        i32 = dict(dtype=torch.int32, device=device)
        self.cfg = config(w)
        S = moe_send_rows(self.cfg)
        self.logits = torch.empty(N, E, dtype=torch.float32, device=device)
        self.topk_idx = torch.empty(N, k, **i32)
        self.topk_w = torch.empty(N, k, dtype=torch.float32, device=device)
        self.xperm = torch.empty(S, d, dtype=dt, device=device)
        self.yperm = torch.empty(S, d, dtype=dt, device=device)
        self.yshared = torch.empty(N, d, dtype=dt, device=device) if w.shared_d_ff else None
        self.out = torch.empty(N, d, dtype=dt, device=device)
        self.expert_counts = torch.empty(E, **i32)
        self.kept_counts = torch.empty(E, **i32)
        self.expert_start = torch.empty(E, **i32)
        self.rank_counts = torch.empty(R, **i32)
        self.rank_offsets = torch.empty(R + 1, **i32)
        self.slot_of = torch.empty(N * k, **i32)
        self.perm_src = torch.empty(S, **i32)
        self.num_kept = torch.empty(1, **i32)
        # INT8 payload path: send and return buffers as codes + per-row scales
        self.int8_payload = getattr(w, "payload", "act") == "int8"
        self.xperm_q = self.xscale = self.yperm_q = self.yscale = None
        if self.int8_payload:
            self.xperm_q = torch.empty(S, d, dtype=torch.int8, device=device)
            self.xscale = torch.empty(S, dtype=torch.float32, device=device)
            self.yperm_q = torch.empty(S, d, dtype=torch.int8, device=device)
            self.yscale = torch.empty(S, dtype=torch.float32, device=device)
        nbytes = moe_workspace_size(self.cfg)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.workspace[:256].zero_()          # sticky device status word starts at 0


def with_tokens(cfg, tokens):
    """Copy of a moe_config with another token count: the union of the data-parallel
    replicas' batches, for the bias update over all-reduced counts."""
    c = moe_config.from_buffer_copy(cfg)
    c.tokens = int(tokens)
    return c


def layer_parts(b, inp, bias_step=0.0, stream=None, replicas=1, saved=None):
    """The layer step as three stream-ordered parts: (1) route and dispatch, (2) expert
    FFN and combine, (3) the bias update (None when there is none).  With an INT8
    payload (LayerBuffers of a workload with payload="int8") the send and return
    buffers hold INT8 codes + per-row scales: part 1 is route, dispatch_q8 and
    dequant_rows; part 2 expert FFN, quant_rows and combine_q8.  With data-parallel
    replicas the counts all-reduce goes between part 1 and part 3, and part 3 compares
    the summed counts with the mean load of all `replicas` batches."""
    c = b.cfg

    def send():
        moe_route(c, inp["x"], inp["w_router"], inp["b_router"], inp["sel_bias"], b.logits,
                  b.topk_idx, b.topk_w, b.workspace, stream)
        if b.int8_payload:
            moe_dispatch_q8(c, b.topk_idx, inp["x"], b.xperm_q, b.xscale, b.expert_counts,
                            b.kept_counts, b.expert_start, b.rank_counts, b.rank_offsets,
                            b.slot_of, b.perm_src, b.num_kept, b.workspace, stream)
            moe_dequant_rows(c, b.xperm_q, b.xscale, b.perm_src, b.xperm, stream)
        else:
            moe_dispatch(c, b.topk_idx, inp["x"], b.xperm, b.expert_counts, b.kept_counts,
                         b.expert_start, b.rank_counts, b.rank_offsets, b.slot_of, b.perm_src,
                         b.num_kept, b.workspace, stream)

    def compute_return():
        if saved is not None:   # training: keep h and g|u for the backward
            moe_expert_ffn_save(c, b.xperm, b.expert_start, b.kept_counts, inp["w_gate_up"],
                                inp["w_down"], inp["x"], inp["shared_gate_up"],
                                inp["shared_down"], b.yperm, b.yshared, saved, b.workspace,
                                stream)
        else:
            moe_expert_ffn(c, b.xperm, b.expert_start, b.kept_counts, inp["w_gate_up"],
                           inp["w_down"], inp["x"], inp["shared_gate_up"], inp["shared_down"],
                           b.yperm, b.yshared, b.workspace, stream)
        if b.int8_payload:
            moe_quant_rows(c, b.yperm, b.perm_src, b.yperm_q, b.yscale, stream)
            moe_combine_q8(c, b.yperm_q, b.yscale, b.slot_of, b.topk_w, inp["x"], b.yshared,
                           b.out, stream)
        else:
            moe_combine(c, b.yperm, b.slot_of, b.topk_w, inp["x"], b.yshared, b.out, stream)

    update = None
    if bias_step and inp["sel_bias"] is not None:
        cb = with_tokens(c, c.tokens * replicas) if replicas > 1 else c

        def update():
            moe_bias_update(cb, b.expert_counts, inp["sel_bias"], bias_step, stream)
    return send, compute_return, update


def run_layer(b, inp, bias_step=0.0, stream=None, reduce_counts=None, replicas=1, saved=None):
    """One pass of the layer path through the C ABI: route, dispatch, expert FFN,
    combine, and (if bias_step) the selection-bias update (see layer_parts).

    Data-parallel replicas (each its own token batch, the same layer): the bias update
    needs the load of every replica's batch.  `reduce_counts(expert_counts)` sums the
    routed counts over the replicas in place (an all-reduce; it may return a handle
    whose .wait() orders it before the bias update, so that it overlaps the expert
    FFN), and the sign rule then compares the summed counts with the mean load of all
    `replicas` batches.  b.expert_counts holds the summed counts afterwards.  With
    `saved` (moe_saved_size bytes) the expert FFN also keeps its activations there for
    run_layer_backward."""
    send, compute_return, update = layer_parts(b, inp, bias_step, stream, replicas, saved)
    send()
    handle = None
    if update is not None and reduce_counts is not None:
        if stream is None:
            handle = reduce_counts(b.expert_counts)
        else:
            with torch.cuda.stream(stream):
                handle = reduce_counts(b.expert_counts)
    compute_return()
    if update is not None:
        if handle is not None:
            if stream is None:
                handle.wait()
            else:
                with torch.cuda.stream(stream):
                    handle.wait()
        update()
    return b.out
