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
With a capacity-padded send buffer every chunk is one expert's whole block of C rows at
a fixed offset, so the plan is fixed (StaticExchangePlan) and a step moves no counts at
all.  Both exchanges and the local experts run in steps over source groups (ring
distances, the rank's own rows first), overlapped: group g's expert FFN starts when
group g's rows have landed and its results go back while group g+1 computes
(overlapped_exchange; on one device, run_layer_loopback(overlap=True) runs the copies on
a second stream ordered by events).
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


def source_groups(R, G):
    """Ring distances 0..R-1 split into G contiguous runs (the first holds distance 0, a
    rank's own rows).  In step g a rank receives from the ranks (me - j) mod R and sends
    to the ranks (me + j) mod R, for every distance j of run g."""
    G = max(1, min(int(G), R))
    return [list(range(g * R // G, (g + 1) * R // G)) for g in range(G)]


class ExchangePlan:
    """Chunks of both exchanges for rank `me`, from kept[src, e] (rows that rank src
    keeps for expert e, every rank's counts, host integers).

      send_chunks  (dst, e, offset in the send buffer, rows): this rank's rows for
                   expert e, in send order (dst ascending, e ascending within dst)
      recv_chunks  (src, e, offset in the receive buffer, rows)
      local_experts, local_start, local_kept: the receive buffer's expert segments
      recv_rows, send_rows

    With groups=G the exchange and the expert FFN run in G steps over source groups
    (source_groups): the receive buffer is group-major, expert-major within a group,
    sources ascending within an expert, so each step's rows form one block
    (group_rows[g]) whose expert segments (group_start[g], group_kept[g], relative to
    the block) feed one grouped expert-FFN call while the next step's rows travel.
    groups=1 is the plain expert-major layout.
    """

    def __init__(self, kept, E, R, rank_map, me, groups=1):
        kept = np.asarray(kept, dtype=np.int64).reshape(R, E)
        self._build(lambda src, e: int(kept[src, e]), E, R, rank_map, me, groups,
                    send_offsets=None)

    def _build(self, count, E, R, rank_map, me, groups, send_offsets):
        self.me, self.E, self.R = me, E, R
        self.dist_groups = source_groups(R, groups)
        self.G = len(self.dist_groups)
        step_of_dist = {j: g for g, js in enumerate(self.dist_groups) for j in js}
        self.send_chunks, self.send_step = [], []
        off = 0
        for dst in range(R):
            for e in experts_of_rank(dst, E, R, rank_map):
                n = count(me, e)
                o = off if send_offsets is None else send_offsets[e]
                self.send_chunks.append((dst, e, o, n))
                self.send_step.append(step_of_dist[(dst - me) % R])
                off += n
        self.send_rows = off
        self.local_experts = experts_of_rank(me, E, R, rank_map)
        self.recv_chunks, self.recv_step = [], []
        self.group_rows, self.group_start, self.group_kept = [], [], []
        self.group_sources = []
        off = 0
        for g, js in enumerate(self.dist_groups):
            srcs = sorted((me - j) % R for j in js)
            self.group_sources.append(srcs)
            g0 = off
            starts, kepts = [], []
            for e in self.local_experts:
                starts.append(off - g0)
                for src in srcs:
                    n = count(src, e)
                    self.recv_chunks.append((src, e, off, n))
                    self.recv_step.append(g)
                    off += n
                kepts.append(off - g0 - starts[-1])
            self.group_rows.append((g0, off))
            self.group_start.append(starts)
            self.group_kept.append(kepts)
        self.recv_rows = off
        # expert segments of the whole receive buffer: only with one group (the plain
        # layout) is every expert one contiguous segment
        if self.G == 1:
            self.local_start = list(self.group_start[0])
            self.local_kept = list(self.group_kept[0])
        else:
            self.local_start = self.local_kept = None

    def send_offset(self, dst, e):
        for (r, ee, off, n) in self.send_chunks:
            if r == dst and ee == e:
                return off, n
        raise KeyError((dst, e))


class StaticExchangePlan(ExchangePlan):
    """The plan for a capacity-padded send buffer (MOE_DISPATCH_CAPACITY_PADDED): every
    (rank, expert) chunk is the expert's whole block of C rows at a fixed offset, kept or
    not, so the plan, the split sizes and the receive layout are known before any
    routing and no counts travel to the host.  Rows of a block past the expert's kept
    count hold no assignment: the receiver's expert FFN runs over them (whole blocks, as
    in GShard) and their results are returned to send rows that the combine never reads.
    send_offsets: the dispatch's expert_start (expert e's block at its send position
    times C)."""

    def __init__(self, E, R, rank_map, me, C, groups=1):
        pos = [e for r in range(R) for e in experts_of_rank(r, E, R, rank_map)]
        offsets = {e: i * C for i, e in enumerate(pos)}
        self.C = C
        self._build(lambda src, e: C, E, R, rank_map, me, groups, send_offsets=offsets)


def gather_kept(kept_counts, group=None):
    """Every rank's kept counts [R, E] on the host (an all-gather, then one copy)."""
    import torch.distributed as dist
    R = dist.get_world_size(group)
    out = [torch.empty_like(kept_counts) for _ in range(R)]
    dist.all_gather(out, kept_counts, group=group)
    return torch.stack(out).cpu().numpy()


def _parts(buf):
    return tuple(buf) if isinstance(buf, (tuple, list)) else (buf,)


def exchange_dist(plan, send_buf, recv_buf, reverse=False, group=None, step=None, wait=True):
    """One exchange through torch.distributed.  Forward: send_buf (this rank's send
    buffer) -> recv_buf (the plan's receive layout).  reverse=True: the results in
    recv_buf go back to their source ranks, landing in send_buf at the rows they came
    from.  step: only that source group's chunks (None: all).  Chunks to and from this
    rank itself are copies on the current stream.  wait=True returns after every
    operation completed; wait=False returns the operations' work handles (with NCCL,
    work.wait() orders the current CUDA stream after the transfer without blocking the
    host)."""
    import torch.distributed as dist
    me = plan.me
    sends, recvs = _parts(send_buf), _parts(recv_buf)
    assert len(sends) == len(recvs)
    out_chunks = [c for c, g in zip(plan.send_chunks, plan.send_step) if step is None or g == step]
    in_chunks = [c for c, g in zip(plan.recv_chunks, plan.recv_step) if step is None or g == step]
    incoming = {(src, e): (off, n) for (src, e, off, n) in plan.recv_chunks}
    # rank-to-rank order of the messages: both sides walk one pair's chunks in expert
    # order, and the parts of a chunk in tuple order
    ops = []
    if not reverse:
        for (dst, e, off, n) in out_chunks:
            if n and dst != me:
                ops += [dist.P2POp(dist.isend, t[off:off + n], dst, group) for t in sends]
        for (src, e, off, n) in in_chunks:
            if n and src != me:
                ops += [dist.P2POp(dist.irecv, t[off:off + n], src, group) for t in recvs]
    else:
        for (src, e, off, n) in in_chunks:
            if n and src != me:
                ops += [dist.P2POp(dist.isend, t[off:off + n], src, group) for t in recvs]
        for (dst, e, off, n) in out_chunks:
            if n and dst != me:
                ops += [dist.P2POp(dist.irecv, t[off:off + n], dst, group) for t in sends]
    for (dst, e, off, n) in out_chunks:      # this rank's own experts
        if n and dst == me:
            roff, rn = incoming[(me, e)]
            assert rn == n
            for ts, tr in zip(sends, recvs):
                if not reverse:
                    tr[roff:roff + n].copy_(ts[off:off + n])
                else:
                    ts[off:off + n].copy_(tr[roff:roff + n])
    works = dist.batch_isend_irecv(ops) if ops else []
    if wait:
        for req in works:
            req.wait()
        return []
    return works


def exchange_loopback(plans, send_bufs, recv_bufs, reverse=False, step=None):
    """Both exchanges for ranks held in one process: every chunk is a copy (on the
    current stream).  step: only that source group's chunks of every receiver."""
    for me, plan in enumerate(plans):
        for (src, e, roff, n), g in zip(plan.recv_chunks, plan.recv_step):
            if not n or (step is not None and g != step):
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
    buffers.

    groups: the exchange and the local expert FFN run in that many steps over source
    groups (ExchangePlan), so that one group's expert FFN overlaps the next group's
    transfer and the previous group's results travelling back.
    static: the send buffer is capacity-padded (the workload's dispatch_mode is
    MOE_DISPATCH_CAPACITY_PADDED, with a capacity factor) and the plan is the fixed
    StaticExchangePlan, built once here, with its segment tables on the device: a layer
    step then needs no count exchange and no host synchronisation.
    Otherwise recv_capacity rows are reserved, by default the worst case (every rank
    sends every row here, R * tokens * top_k); a step whose plan needs more raises
    before any copy."""

    def __init__(self, w, rank, inp, device="cuda", recv_capacity=None, groups=1, static=False):
        if w.rank_map != RANK_ROUND_ROBIN and w.num_experts % w.num_ranks:
            raise ValueError("contiguous expert blocks need num_experts % num_ranks == 0")
        self.w, self.rank, self.inp = w, rank, inp
        self.b = moe.LayerBuffers(w, device)
        R, E, N, k, d = w.num_ranks, w.num_experts, w.tokens, w.top_k, w.hidden
        self.local = experts_of_rank(rank, E, R, w.rank_map)
        self.groups, self.static = int(groups), bool(static)
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
        self.static_plan = None
        if self.static:
            if getattr(w, "dispatch_mode", 0) != 1 or not w.capacity_factor > 0:
                raise ValueError("a static exchange needs the capacity-padded dispatch layout")
            C = moe.moe_send_rows(self.b.cfg) // E
            self.static_plan = StaticExchangePlan(E, R, w.rank_map, rank, C, self.groups)
            cap = max(self.static_plan.recv_rows, 1)
        else:
            cap = max(R * N * k if recv_capacity is None else int(recv_capacity), 1)
        self.recv_capacity = cap
        self.recv_x = torch.empty(cap, d, dtype=w.torch_dtype, device=device)
        self.recv_y = torch.empty(cap, d, dtype=w.torch_dtype, device=device)
        self.int8 = getattr(w, "payload", "act") == "int8"
        if self.int8:
            # codes + scales travel, with the source's perm_src of each row: a received
            # row holds an assignment iff that value is >= 0 (padding rows of a
            # capacity-padded block do not)
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
        G = len(source_groups(R, self.groups))
        # per source group: its experts' segment starts and row counts in the group's block
        self.g_start = torch.zeros(G, len(self.local), dtype=torch.int32, device=device)
        self.g_kept = torch.zeros(G, len(self.local), dtype=torch.int32, device=device)
        self.zero_counts = torch.zeros(E, dtype=torch.int32, device=device)
        if self.static:
            self.load_plan_tables(self.static_plan)

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
    # receive buffers (activations, or INT8 codes + scales + the rows' perm_src)
    def send_rows(self):
        return (self.b.xperm_q, self.b.xscale, self.b.perm_src) if self.int8 else self.b.xperm

    def return_rows(self):
        return (self.b.yperm_q, self.b.yscale) if self.int8 else self.b.yperm

    def received_rows(self):
        return (self.recv_xq, self.recv_xs, self.recv_valid) if self.int8 else self.recv_x

    def result_rows(self):
        return (self.recv_yq, self.recv_ys) if self.int8 else self.recv_y

    def check_plan(self, plan):
        if plan.recv_rows > self.recv_capacity:
            raise ValueError(f"rank {self.rank} would receive {plan.recv_rows} rows; its "
                             f"receive buffers hold {self.recv_capacity}")

    def load_plan_tables(self, plan, stream=None):
        """The plan's per-group segment tables into device memory, on the stream the
        expert kernels run on (so neither this step's kernels nor the previous step's
        can see them half written)."""
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            self.g_start.copy_(torch.tensor(plan.group_start, dtype=torch.int32))
            self.g_kept.copy_(torch.tensor(plan.group_kept, dtype=torch.int32))

    def local_ffn(self, plan, stream=None, step=0):
        """The local experts on one source group's block of the receive buffer
        (recv_x -> recv_y); with an INT8 payload the received codes are dequantised
        first and the results quantised after.  The segment tables come from
        load_plan_tables."""
        g0, g1 = plan.group_rows[step]
        if g1 == g0:
            return
        # the kernel choice reads the average rows per expert from the configuration
        cfg = moe.config(replace(self.local_w, tokens=g1 - g0))
        rx, ry = self.recv_x[g0:g1], self.recv_y[g0:g1]
        if self.int8:
            moe.moe_dequant_rows(cfg, self.recv_xq[g0:g1], self.recv_xs[g0:g1],
                                 self.recv_valid[g0:g1], rx, stream)
        moe.moe_expert_ffn(cfg, rx, self.g_start[step], self.g_kept[step], self.w_gate_up,
                           self.w_down, None, None, None, ry, None, self.local_ws, stream)
        if self.int8:
            moe.moe_quant_rows(cfg, ry, self.recv_valid[g0:g1], self.recv_yq[g0:g1],
                               self.recv_ys[g0:g1], stream)

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


def overlapped_exchange(plan, send_buf, recv_buf, return_buf, result_buf, compute,
                        group=None):
    """The overlapped schedule of both exchanges around the local experts: every source
    group's receives (and this rank's sends) are issued first; then for each group in
    turn, wait for its rows, compute(g) (the local experts on group g's block), and send
    its results back without waiting.  Returns the return transfers' work handles, to
    wait on before the combine."""
    G = plan.G
    fwd = [exchange_dist(plan, send_buf, recv_buf, group=group, step=g, wait=False)
           for g in range(G)]
    back = []
    for g in range(G):
        for wk in fwd[g]:
            wk.wait()
        compute(g)
        back.append(exchange_dist(plan, return_buf, result_buf, reverse=True, group=group,
                                  step=g, wait=False))
    return [wk for ws in back for wk in ws]


def _plans(ranks):
    """Every rank's plan: the fixed ones, or one from every rank's kept counts (one copy
    of the counts to the host), checked against every rank's receive capacity."""
    if ranks[0].static:
        return [r.static_plan for r in ranks]
    R = len(ranks)
    kept = torch.stack([r.b.kept_counts for r in ranks]).cpu().numpy()
    w0 = ranks[0].w
    plans = [ExchangePlan(kept, w0.num_experts, R, w0.rank_map, me, r.groups)
             for me, r in enumerate(ranks)]
    for r, plan in zip(ranks, plans):
        r.check_plan(plan)
    return plans


def run_layer_loopback(ranks, bias_step=0.0, overlap=False):
    """The expert-parallel layer for ranks held in one process (one device): route and
    dispatch on every rank, the exchange, every rank's local experts, the return
    exchange, the shared expert and the combine on every rank, and the bias update
    from the summed counts (the sum stands in for the all-reduce).  Returns the plans.

    overlap=True runs the exchanges' copies on a second stream, source group by source
    group: group g's expert FFN (on the current stream) waits only for group g's copies,
    and its results start back while the next group computes.  Streams and events order
    everything; no kernel waits on another."""
    R = len(ranks)
    for r in ranks:
        r.route_dispatch()
    plans = _plans(ranks)
    if not ranks[0].static:
        for r, plan in zip(ranks, plans):
            r.load_plan_tables(plan)
    G = plans[0].G
    sends = [r.send_rows() for r in ranks]
    recvs = [r.received_rows() for r in ranks]
    rets = [r.return_rows() for r in ranks]
    ress = [r.result_rows() for r in ranks]
    if not overlap:
        for g in range(G):
            exchange_loopback(plans, sends, recvs, step=g)
        for g in range(G):
            for r, plan in zip(ranks, plans):
                r.local_ffn(plan, step=g)
        for g in range(G):
            exchange_loopback(plans, rets, ress, reverse=True, step=g)
        for r in ranks:
            r.shared_ffn()
    else:
        comp = torch.cuda.current_stream()
        copy = torch.cuda.Stream(device=comp.device)
        ready = torch.cuda.Event()
        ready.record(comp)                    # every rank's send buffer is written
        copy.wait_event(ready)
        landed = [torch.cuda.Event() for _ in range(G)]
        with torch.cuda.stream(copy):
            for g in range(G):
                exchange_loopback(plans, sends, recvs, step=g)
                landed[g].record(copy)
        computed = [torch.cuda.Event() for _ in range(G)]
        for g in range(G):
            comp.wait_event(landed[g])
            for r, plan in zip(ranks, plans):
                r.local_ffn(plan, step=g)
            computed[g].record(comp)
            with torch.cuda.stream(copy):
                copy.wait_event(computed[g])
                exchange_loopback(plans, rets, ress, reverse=True, step=g)
        for r in ranks:
            r.shared_ffn()                   # overlaps the returns still in flight
        back = torch.cuda.Event()
        back.record(copy)
        comp.wait_event(back)
    for r in ranks:
        r.combine()
    w0 = ranks[0].w
    if bias_step and ranks[0].inp["sel_bias"] is not None:
        total = torch.stack([r.b.expert_counts for r in ranks]).sum(0).to(torch.int32)
        cb = moe.with_tokens(ranks[0].b.cfg, w0.tokens * R)
        moe.moe_bias_update(cb, total, ranks[0].inp["sel_bias"], bias_step)
    return plans


def run_layer_dist(rank_layer, group=None, bias_step=0.0):
    """This rank's part of the expert-parallel layer over torch.distributed (one rank
    per GPU, every rank with the same receive capacity and groups): route and dispatch,
    the plan (fixed, or from every rank's kept counts), then per source group the
    transfer, the local experts and the return, overlapped: every group's receives are
    issued first, group g's expert FFN waits only for its own rows, and its results are
    sent back while the next group computes; the shared expert runs while the last
    results travel.  Then the combine and the bias update from the all-reduced counts.
    With NCCL the waits order the CUDA stream without blocking the host.  Returns the
    plan."""
    import torch.distributed as dist
    r = rank_layer
    w = r.w
    r.route_dispatch()
    if r.static:
        plan = r.static_plan                 # no counts cross, nothing waits on the host
    else:
        kept = gather_kept(r.b.kept_counts, group)
        plan = ExchangePlan(kept, w.num_experts, w.num_ranks, w.rank_map, r.rank, r.groups)
        # every rank holds every rank's counts, so with the same receive capacity on every
        # rank all ranks take the same decision here and none is left waiting in an exchange
        for other in range(w.num_ranks):
            r.check_plan(ExchangePlan(kept, w.num_experts, w.num_ranks, w.rank_map, other,
                                      r.groups))
        r.load_plan_tables(plan)
    back = overlapped_exchange(plan, r.send_rows(), r.received_rows(), r.return_rows(),
                               r.result_rows(), lambda g: r.local_ffn(plan, step=g), group)
    r.shared_ffn()                           # overlaps the results still travelling
    for wk in back:
        wk.wait()
    r.combine()
    if bias_step and r.inp["sel_bias"] is not None:
        # summed into a copy: this rank's own routing counts stay in b.expert_counts
        total = r.b.expert_counts.clone()
        dist.all_reduce(total, group=group)
        cb = moe.with_tokens(r.b.cfg, w.tokens * w.num_ranks)
        moe.moe_bias_update(cb, total, r.inp["sel_bias"], bias_step)
    return plan
