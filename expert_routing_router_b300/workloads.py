"""The five synthetic MoE-layer workloads and their seeded input generators.

This module only draws random numbers with the shapes and distributions of the
workloads; it holds none of the layer's arithmetic.  Tests, the benchmark and the
smoke check take their inputs from here, and the same tensors are handed both to
the CUDA library and (copied to the host) to the CPU oracle.

Workloads (named by what they are):
  tiny_top2_f32       4096 x 512, 8 experts, top-2 softmax renormalised, fp32,
                      4 ranks; reproduces the routing example of the Ultralytics
                      glossary page "Expert Parallelism" (seed 0, CPU generator,
                      nn.Linear(512, 8) default init).
  switch_top1_bf16    16384 x 1024, 32 experts, top-1, capacity factor 1.25, 8 ranks.
  gshard_top2_skewed  32768 x 2048, 64 experts, top-2, per-expert logit offset
                      N(0, 1.5) folded into the router bias, capacity 1.25, 16 ranks.
  dsv3_prefill        8192 x 7168, 256 experts, sigmoid + selection bias N(0, 0.1),
                      8 groups / top-4 groups, top-8, renormalised, shared expert,
                      64 ranks, bias update step 1e-3.
  dsv3_decode         the same layer at 1, 8, 64, 128, 512 tokens, 40 ranks
                      assigned round-robin.
  gshard_top2_padded  the GShard-shaped layer with the capacity-padded [E, C] send
                      buffer and choice-major capacity priority.
  dsv3_prefill_int8   the DeepSeek-V3 prefill layer with the all-to-all payload (send
                      and return buffers) as INT8 codes + per-row fp32 scales.
"""
from dataclasses import dataclass, replace
import math

import torch

SCORE_SOFTMAX = 0
SCORE_SIGMOID = 1
RANK_CONTIGUOUS = 0
RANK_ROUND_ROBIN = 1


@dataclass(frozen=True)
class Workload:
    name: str
    tokens: int
    hidden: int
    num_experts: int
    top_k: int
    num_ranks: int
    rank_map: int
    score_fn: int
    normalize_topk: bool
    num_groups: int
    topk_groups: int
    capacity_factor: float
    d_ff: int
    shared_d_ff: int
    act_dtype: str            # "f32" or "bf16"
    router_offset_std: float  # per-expert logit offset folded into the router bias
    sel_bias_std: float       # selection-only bias (sigmoid scoring)
    bias_step: float          # bias-update step (0 = no update in the step)
    expert_std: float = 0.02
    dispatch_mode: int = 0    # 0 packed token-order capacity, 1 capacity-padded choice-major
    payload: str = "act"      # all-to-all payload: "act" (activation dtype) or "int8"

    def with_tokens(self, n):
        return replace(self, tokens=n, name=f"{self.name.split('@')[0]}@{n}")

    @property
    def torch_dtype(self):
        return torch.float32 if self.act_dtype == "f32" else torch.bfloat16


TINY_TOP2_F32 = Workload("tiny_top2_f32", 4096, 512, 8, 2, 4, RANK_CONTIGUOUS, SCORE_SOFTMAX,
                         True, 1, 1, 0.0, 256, 0, "f32", 0.0, 0.0, 0.0)
SWITCH_TOP1 = Workload("switch_top1_bf16", 16384, 1024, 32, 1, 8, RANK_CONTIGUOUS, SCORE_SOFTMAX,
                       False, 1, 1, 1.25, 2048, 0, "bf16", 0.0, 0.0, 0.0)
GSHARD_TOP2 = Workload("gshard_top2_skewed", 32768, 2048, 64, 2, 16, RANK_CONTIGUOUS,
                       SCORE_SOFTMAX, False, 1, 1, 1.25, 1408, 0, "bf16", 1.5, 0.0, 0.0)
GSHARD_TOP2_PADDED = replace(GSHARD_TOP2, name="gshard_top2_padded", dispatch_mode=1)
DSV3_PREFILL = Workload("dsv3_prefill", 8192, 7168, 256, 8, 64, RANK_CONTIGUOUS, SCORE_SIGMOID,
                        True, 8, 4, 0.0, 2048, 2048, "bf16", 0.0, 0.1, 1e-3)
DSV3_PREFILL_INT8 = replace(DSV3_PREFILL, name="dsv3_prefill_int8", payload="int8")
DSV3_DECODE = replace(DSV3_PREFILL, name="dsv3_decode", tokens=512, num_ranks=40,
                      rank_map=RANK_ROUND_ROBIN)
DECODE_TOKENS = (1, 8, 64, 128, 512)

WORKLOADS = {w.name: w for w in (TINY_TOP2_F32, SWITCH_TOP1, GSHARD_TOP2, GSHARD_TOP2_PADDED,
                                 DSV3_PREFILL, DSV3_PREFILL_INT8, DSV3_DECODE)}


def _normal_(t, std, gen, chunk_rows=64):
    """Fill t with N(0, std) in row chunks (keeps fp32 temporaries small)."""
    flat = t.view(t.shape[0], -1) if t.dim() > 1 else t.view(1, -1)
    for r0 in range(0, flat.shape[0], chunk_rows):
        rows = flat[r0:r0 + chunk_rows]
        tmp = torch.randn(rows.shape, generator=gen, device=t.device, dtype=torch.float32)
        rows.copy_(tmp.mul_(std))
    return t


def make_inputs(w: Workload, seed: int = 0, device="cpu", with_experts=True):
    """Draw every input of the layer for workload `w`.

    Returns a dict of tensors on `device`:
      x [N, d] act dtype, w_router [E, d] fp32, b_router [E] fp32,
      sel_bias [E] fp32 or None, w_gate_up [E, 2F, d], w_down [E, d, F],
      shared_gate_up [2Fs, d] / shared_down [d, Fs] or None (act dtype).

    The tiny fp32 workload draws from torch's global CPU generator in the order of
    the glossary page's example (hidden states, then nn.Linear's default init of
    weight and bias), then the expert weights; everything else draws from a
    dedicated generator on `device`.
    """
    N, d, E = w.tokens, w.hidden, w.num_experts
    dt = w.torch_dtype
    out = {}
    if w.name.startswith("tiny_top2_f32"):
        # the page's example: global CPU generator, hidden states then nn.Linear init
        draw = "cpu"
        torch.manual_seed(seed)
        gen = torch.default_generator
        out["x"] = torch.randn(N, d)
        lin = torch.nn.Linear(d, E)
        out["w_router"] = lin.weight.detach().clone()
        out["b_router"] = lin.bias.detach().clone()
    else:
        draw = device
        gen = torch.Generator(device=draw)
        gen.manual_seed(seed)
        x = torch.empty(N, d, dtype=dt, device=draw)
        _normal_(x, 1.0, gen, chunk_rows=4096)
        out["x"] = x
        bound = 1.0 / math.sqrt(d)
        wr = torch.empty(E, d, dtype=torch.float32, device=draw)
        wr.uniform_(-bound, bound, generator=gen)
        br = torch.empty(E, dtype=torch.float32, device=draw)
        br.uniform_(-bound, bound, generator=gen)
        if w.router_offset_std > 0:
            off = torch.randn(E, generator=gen, device=draw) * w.router_offset_std
            br = br + off
        out["w_router"] = wr
        out["b_router"] = br
    out["sel_bias"] = None
    if w.sel_bias_std > 0:
        out["sel_bias"] = torch.randn(E, generator=gen, device=draw) * w.sel_bias_std
    out["w_gate_up"] = out["w_down"] = None
    out["shared_gate_up"] = out["shared_down"] = None
    if with_experts:
        F, Fs = w.d_ff, w.shared_d_ff
        wgu = torch.empty(E, 2 * F, d, dtype=dt, device=draw)
        wd = torch.empty(E, d, F, dtype=dt, device=draw)
        for e in range(E):
            _normal_(wgu[e], w.expert_std, gen, chunk_rows=1024)
            _normal_(wd[e], w.expert_std, gen, chunk_rows=1024)
        out["w_gate_up"], out["w_down"] = wgu, wd
        if Fs > 0:
            sgu = torch.empty(2 * Fs, d, dtype=dt, device=draw)
            sd = torch.empty(d, Fs, dtype=dt, device=draw)
            _normal_(sgu, w.expert_std, gen, chunk_rows=1024)
            _normal_(sd, w.expert_std, gen, chunk_rows=1024)
            out["shared_gate_up"], out["shared_down"] = sgu, sd
    if str(draw) != str(device):
        out = {k: (None if v is None else v.to(device)) for k, v in out.items()}
    return out


def make_tokens(w: Workload, n_tokens: int, seed: int, device="cpu"):
    """Fresh hidden states x [n_tokens, d] for an existing layer (decode sweep)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 7919 * n_tokens)
    x = torch.empty(n_tokens, w.hidden, dtype=w.torch_dtype, device=device)
    return _normal_(x, 1.0, gen, chunk_rows=4096)
