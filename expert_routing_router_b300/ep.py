"""Expert parallelism: the all-to-all exchange around the expert FFN.

Ultralytics glossary "Expert Parallelism", section "How tokens move between GPUs":
each device routes its own tokens (step 1), sends every kept (token, expert) row to
the device that holds the expert (step 2), runs its local experts on what it received
(step 3) and sends the results back to the tokens' home devices, where they are
weighted and summed (step 4).  The example on that page counts, per device, the rows
each device receives; those counts are the split sizes of the two exchanges here.

The dispatch already writes the send buffer in the order an exchange sends it: rank
(the expert's owner) ascending, expert ascending within a rank, token order within an
expert, so the rows for one (destination, expert) pair are one contiguous chunk at
expert_start[e].  The receiver lays its rows out expert-major (local experts
ascending, source ranks ascending within an expert, each source's rows in its token
order), so every local expert is one contiguous segment and the grouped expert FFN
runs on the receive buffer unchanged.  The return exchange sends each result chunk
back to the position its row came from, so the source's return buffer has its send
buffer's layout and the combine runs on it unchanged.

Two transports move the chunks:
  exchange_dist      torch.distributed point-to-point operations, one pair of
                     operations per non-empty (peer, expert) chunk, issued as one batch
                     (NCCL between GPUs, gloo on CPU); a rank's chunks to itself are
                     copies.
  exchange_loopback  every rank's buffers in one process (one device): the chunks are
                     copies.  It runs the whole expert-parallel layer on one GPU, ranks
                     one after another, with nothing waiting on another rank.

The chunk sizes come from every rank's kept counts, gathered to the host once per step
(ExchangePlan): the point-to-point sizes must be known where the operations are issued.
The shared expert runs on the tokens' home rank (it sees every token) and is not sent.
A buffer argument of the exchanges may be a tuple of row-aligned tensors (an INT8
payload: codes [rows, d] int8 and scales [rows] fp32), moved chunk by chunk together.
With a workload whose payload is "int8", the rank layer sends codes and scales both
ways (moe_dispatch_q8 on the source, moe_dequant_rows and moe_quant_rows around the
local experts on the receiver, moe_combine_q8 back on the source).
"""
from dataclasses import replace

import numpy as np
import torch

from . import moe

RANK_CONTIGUOUS = 0
RANK_ROUND_ROBIN = 1


def experts_of_rank(r, E, R, rank_map):
    """Experts held by rank r, ascending (contiguous blocks of E/R, or e mod R == r)."""
    if rank_map == RANK_ROUND_ROBIN:
        return list(range(r, E, R))
    per = E // R
    return list(range(r * per, (r + 1) * per))


class ExchangePlan:
    """Chunks of both exchanges for rank `me`, from kept[src, e] (rows that rank src
    keeps for expert e, every rank's counts, host integers).

      send_chunks  (dst, e, offset in the send buffer, rows): this rank's rows for
                   expert e, in send order (dst ascending, e ascending within dst)
      recv_chunks  (src, e, offset in the receive buffer, rows): expert-major
      local_experts, local_start, local_kept: the receive buffer's expert segments
      recv_rows, send_rows
    """

    def __init__(self, kept, E, R, rank_map, me):
        kept = np.asarray(kept, dtype=np.int64).reshape(R, E)
        self.me, self.E, self.R = me, E, R
        self.send_chunks = []
        off = 0
        for dst in range(R):
            for e in experts_of_rank(dst, E, R, rank_map):
                n = int(kept[me, e])
                self.send_chunks.append((dst, e, off, n))
                off += n
        self.send_rows = off
        self.local_experts = experts_of_rank(me, E, R, rank_map)
        self.recv_chunks, self.local_start, self.local_kept = [], [], []
        off = 0
        for e in self.local_experts:
            self.local_start.append(off)
            for src in range(R):
                n = int(kept[src, e])
                self.recv_chunks.append((src, e, off, n))
                off += n
            self.local_kept.append(off - self.local_start[-1])
        self.recv_rows = off

    def send_offset(self, dst, e):
        for (r, ee, off, n) in self.send_chunks:
            if r == dst and ee == e:
                return off, n
        raise KeyError((dst, e))


def gather_kept(kept_counts, group=None):
    """Every rank's kept counts [R, E] on the host (an all-gather, then one copy)."""
    import torch.distributed as dist
    R = dist.get_world_size(group)
    out = [torch.empty_like(kept_counts) for _ in range(R)]
    dist.all_gather(out, kept_counts, group=group)
    return torch.stack(out).cpu().numpy()


def _parts(buf):
    return tuple(buf) if isinstance(buf, (tuple, list)) else (buf,)


def exchange_dist(plan, send_buf, recv_buf, reverse=False, group=None):
    """One exchange through torch.distributed.  Forward: send_buf (this rank's send
    buffer) -> recv_buf (expert-major).  reverse=True: the results in recv_buf go back
    to their source ranks, landing in send_buf at the rows they came from.  Chunks to
    and from this rank itself are copies.  Returns after every operation completed."""
    import torch.distributed as dist
    me = plan.me
    sends, recvs = _parts(send_buf), _parts(recv_buf)
    assert len(sends) == len(recvs)
    # rank-to-rank order of the messages: both sides walk one pair's chunks in expert
    # order, and the parts of a chunk in tuple order
    outgoing = [(dst, e, off, n) for (dst, e, off, n) in plan.send_chunks]
    incoming = {(src, e): (off, n) for (src, e, off, n) in plan.recv_chunks}
    ops = []
    if not reverse:
        for (dst, e, off, n) in outgoing:
            if n and dst != me:
                ops += [dist.P2POp(dist.isend, t[off:off + n], dst, group) for t in sends]
        for (src, e, off, n) in plan.recv_chunks:
            if n and src != me:
                ops += [dist.P2POp(dist.irecv, t[off:off + n], src, group) for t in recvs]
    else:
        for (src, e, off, n) in plan.recv_chunks:
            if n and src != me:
                ops += [dist.P2POp(dist.isend, t[off:off + n], src, group) for t in recvs]
        for (dst, e, off, n) in outgoing:
            if n and dst != me:
                ops += [dist.P2POp(dist.irecv, t[off:off + n], dst, group) for t in sends]
    for (dst, e, off, n) in outgoing:        # this rank's own experts
        if n and dst == me:
            roff, rn = incoming[(me, e)]
            assert rn == n
            for ts, tr in zip(sends, recvs):
                if not reverse:
                    tr[roff:roff + n].copy_(ts[off:off + n])
                else:
                    ts[off:off + n].copy_(tr[roff:roff + n])
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()


def exchange_loopback(plans, send_bufs, recv_bufs, reverse=False):
    """Both exchanges for ranks held in one process: every chunk is a copy."""
    for me, plan in enumerate(plans):
        for (src, e, roff, n) in plan.recv_chunks:
            if not n:
                continue
            soff, sn = plans[src].send_offset(me, e)
            assert sn == n
            for ts, tr in zip(_parts(send_bufs[src]), _parts(recv_bufs[me])):
                if not reverse:
                    tr[roff:roff + n].copy_(ts[soff:soff + n])
                else:
                    ts[soff:soff + n].copy_(tr[roff:roff + n])


class RankLayer:
    """One rank of an expert-parallel layer: its LayerBuffers (the workload's
    num_ranks is the number of ranks), its local experts' weights, and the receive
    buffers: recv_capacity rows, by default the worst case (every rank sends every row
    here, R * tokens * top_k); a step whose plan needs more raises before any copy."""

    def __init__(self, w, rank, inp, device="cuda", recv_capacity=None):
        if w.rank_map != RANK_ROUND_ROBIN and w.num_experts % w.num_ranks:
            raise ValueError("contiguous expert blocks need num_experts % num_ranks == 0")
        self.w, self.rank, self.inp = w, rank, inp
        self.b = moe.LayerBuffers(w, device)
        R, E, N, k, d = w.num_ranks, w.num_experts, w.tokens, w.top_k, w.hidden
        self.local = experts_of_rank(rank, E, R, w.rank_map)
        # this rank's experts only (an expert-parallel rank stores no other weights):
        # a block of the stacked weights, or a gathered copy for round-robin ownership
        if w.rank_map == RANK_ROUND_ROBIN:
            idx = torch.tensor(self.local, dtype=torch.long, device=device)
            self.w_gate_up = inp["w_gate_up"].index_select(0, idx).contiguous()
            self.w_down = inp["w_down"].index_select(0, idx).contiguous()
        else:
            e0, e1 = self.local[0], self.local[-1] + 1
            self.w_gate_up = inp["w_gate_up"][e0:e1]
            self.w_down = inp["w_down"][e0:e1]
        cap = max(R * N * k if recv_capacity is None else int(recv_capacity), 1)
        self.recv_capacity = cap
        self.recv_x = torch.empty(cap, d, dtype=w.torch_dtype, device=device)
        self.recv_y = torch.empty(cap, d, dtype=w.torch_dtype, device=device)
        self.int8 = getattr(w, "payload", "act") == "int8"
        if self.int8:  # codes + scales travel; every received row holds an assignment
            self.recv_xq = torch.empty(cap, d, dtype=torch.int8, device=device)
            self.recv_xs = torch.empty(cap, dtype=torch.float32, device=device)
            self.recv_yq = torch.empty(cap, d, dtype=torch.int8, device=device)
            self.recv_ys = torch.empty(cap, dtype=torch.float32, device=device)
            self.recv_valid = torch.zeros(cap, dtype=torch.int32, device=device)
        self.local_w = replace(w, name=f"{w.name}.experts{rank}", tokens=cap, top_k=1,
                               num_experts=len(self.local), num_ranks=1, rank_map=0,
                               num_groups=1, topk_groups=1, capacity_factor=0.0,
                               shared_d_ff=0, sel_bias_std=0.0, dispatch_mode=0,
                               payload="act")
        self.local_ws = torch.empty(moe.moe_workspace_size(moe.config(self.local_w)),
                                    dtype=torch.uint8, device=device)
        self.local_ws[:256].zero_()
        self.local_start = torch.zeros(len(self.local), dtype=torch.int32, device=device)
        self.local_kept = torch.zeros(len(self.local), dtype=torch.int32, device=device)
        self.zero_counts = torch.zeros(E, dtype=torch.int32, device=device)

    def route_dispatch(self, stream=None):
        b, inp, c = self.b, self.inp, self.b.cfg
        moe.moe_route(c, inp["x"], inp["w_router"], inp["b_router"], inp["sel_bias"], b.logits,
                      b.topk_idx, b.topk_w, b.workspace, stream)
        if self.int8:
            moe.moe_dispatch_q8(c, b.topk_idx, inp["x"], b.xperm_q, b.xscale, b.expert_counts,
                                b.kept_counts, b.expert_start, b.rank_counts, b.rank_offsets,
                                b.slot_of, b.perm_src, b.num_kept, b.workspace, stream)
        else:
            moe.moe_dispatch(c, b.topk_idx, inp["x"], b.xperm, b.expert_counts, b.kept_counts,
                             b.expert_start, b.rank_counts, b.rank_offsets, b.slot_of,
                             b.perm_src, b.num_kept, b.workspace, stream)

    # the buffers the two exchanges move: this rank's send / return rows, and its
    # receive buffers (activations, or INT8 codes + scales)
    def send_rows(self):
        return (self.b.xperm_q, self.b.xscale) if self.int8 else self.b.xperm

    def return_rows(self):
        return (self.b.yperm_q, self.b.yscale) if self.int8 else self.b.yperm

    def received_rows(self):
        return (self.recv_xq, self.recv_xs) if self.int8 else self.recv_x

    def result_rows(self):
        return (self.recv_yq, self.recv_ys) if self.int8 else self.recv_y

    def check_plan(self, plan):
        if plan.recv_rows > self.recv_capacity:
            raise ValueError(f"rank {self.rank} would receive {plan.recv_rows} rows; its "
                             f"receive buffers hold {self.recv_capacity}")

    def local_ffn(self, plan, stream=None):
        """The local experts on the expert-major receive buffer (recv_x -> recv_y); with
        an INT8 payload the received codes are dequantised first and the results
        quantised after."""
        if not plan.recv_rows:
            return
        # the segment tables are written on the stream the kernels run on, so neither
        # this step's kernels nor the previous step's can see them half written
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            self.local_start.copy_(torch.tensor(plan.local_start, dtype=torch.int32))
            self.local_kept.copy_(torch.tensor(plan.local_kept, dtype=torch.int32))
        # the kernel choice reads the average rows per expert from the configuration
        cfg = moe.config(replace(self.local_w, tokens=plan.recv_rows))
        if self.int8:
            moe.moe_dequant_rows(cfg, self.recv_xq, self.recv_xs, self.recv_valid, self.recv_x,
                                 stream)
        moe.moe_expert_ffn(cfg, self.recv_x, self.local_start, self.local_kept, self.w_gate_up,
                           self.w_down, None, None, None, self.recv_y, None, self.local_ws,
                           stream)
        if self.int8:
            moe.moe_quant_rows(cfg, self.recv_y, self.recv_valid, self.recv_yq, self.recv_ys,
                               stream)

    def shared_ffn(self, stream=None):
        """The shared expert on this rank's own tokens (no routed rows)."""
        b, inp = self.b, self.inp
        if not self.w.shared_d_ff:
            return
        moe.moe_expert_ffn(b.cfg, b.xperm, b.expert_start, self.zero_counts, inp["w_gate_up"],
                           inp["w_down"], inp["x"], inp["shared_gate_up"], inp["shared_down"],
                           b.yperm, b.yshared, b.workspace, stream)

    def combine(self, stream=None):
        b, inp = self.b, self.inp
        if self.int8:
            moe.moe_combine_q8(b.cfg, b.yperm_q, b.yscale, b.slot_of, b.topk_w, inp["x"],
                               b.yshared, b.out, stream)
        else:
            moe.moe_combine(b.cfg, b.yperm, b.slot_of, b.topk_w, inp["x"], b.yshared, b.out,
                            stream)


def run_layer_loopback(ranks, bias_step=0.0):
    """The expert-parallel layer for ranks held in one process (one device): route and
    dispatch on every rank, the exchange, every rank's local experts, the return
    exchange, the shared expert and the combine on every rank, and the bias update
    from the summed counts (the sum stands in for the all-reduce).  Returns the plans."""
    R = len(ranks)
    for r in ranks:
        r.route_dispatch()
    kept = torch.stack([r.b.kept_counts for r in ranks]).cpu().numpy()
    w0 = ranks[0].w
    plans = [ExchangePlan(kept, w0.num_experts, R, w0.rank_map, me) for me in range(R)]
    for r, plan in zip(ranks, plans):
        r.check_plan(plan)
    exchange_loopback(plans, [r.send_rows() for r in ranks], [r.received_rows() for r in ranks])
    for r, plan in zip(ranks, plans):
        r.local_ffn(plan)
    exchange_loopback(plans, [r.return_rows() for r in ranks], [r.result_rows() for r in ranks],
                      reverse=True)
    for r in ranks:
        r.shared_ffn()
        r.combine()
    if bias_step and ranks[0].inp["sel_bias"] is not None:
        total = torch.stack([r.b.expert_counts for r in ranks]).sum(0).to(torch.int32)
        cb = moe.with_tokens(ranks[0].b.cfg, w0.tokens * R)
        moe.moe_bias_update(cb, total, ranks[0].inp["sel_bias"], bias_step)
    return plans


def run_layer_dist(rank_layer, group=None, bias_step=0.0):
    """This rank's part of the expert-parallel layer over torch.distributed (one rank
    per GPU, every rank with the same receive capacity): route and dispatch, gather the
    kept counts, exchange, local experts, return exchange, shared expert, combine, and
    the bias update from the all-reduced counts.  Returns the plan."""
    import torch.distributed as dist
    r = rank_layer
    r.route_dispatch()
    kept = gather_kept(r.b.kept_counts, group)
    w = r.w
    plan = ExchangePlan(kept, w.num_experts, w.num_ranks, w.rank_map, r.rank)
    # every rank holds every rank's counts, so with the same receive capacity on every
    # rank all ranks take the same decision here and none is left waiting in an exchange
    for other in range(w.num_ranks):
        r.check_plan(ExchangePlan(kept, w.num_experts, w.num_ranks, w.rank_map, other))
    exchange_dist(plan, r.send_rows(), r.received_rows(), group=group)
    r.local_ffn(plan)
    exchange_dist(plan, r.return_rows(), r.result_rows(), reverse=True, group=group)
    r.shared_ffn()
    r.combine()
    if bias_step and r.inp["sel_bias"] is not None:
        # summed into a copy: this rank's own routing counts stay in b.expert_counts
        total = r.b.expert_counts.clone()
        dist.all_reduce(total, group=group)
        cb = moe.with_tokens(r.b.cfg, w.tokens * w.num_ranks)
        moe.moe_bias_update(cb, total, r.inp["sel_bias"], bias_step)
    return plan
