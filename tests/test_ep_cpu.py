"""Expert-parallel exchange (host side), on CPU.

The exchange plan is checked against the oracle's dispatch tables (the send buffer
the CUDA dispatch writes has the oracle's layout, bit for bit, per the GPU parity
tests), and the point-to-point exchange itself runs between two gloo ranks on CPU
tensors whose rows name their origin (rank, token, choice, expert): every row must
arrive at the rank that holds its expert, in the expert-major layout, and every
result must come back to the send-buffer row it left from.
"""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from expert_routing_router_b300 import ep


def _routing(rank, N, E, k, seed):
    """Seeded top-k ids of one rank's tokens (distinct experts per token, skewed)."""
    rng = np.random.default_rng(seed + 17 * rank)
    pref = rng.standard_normal(E) * 1.5
    idx = np.empty((N, k), np.int32)
    for t in range(N):
        idx[t] = np.argsort(-(rng.standard_normal(E) + pref), kind="stable")[:k]
    return idx


def _tables(rank, N, E, k, R, rank_map, cf, seed):
    idx = _routing(rank, N, E, k, seed)
    return idx, oracle.dispatch(idx, E, R, rank_map, cf)


def _send_rows(rank, idx, d, k):
    """Send buffer whose kept rows hold (rank, token, choice, expert)."""
    S = d["send_rows"]
    rows = np.full((S, 4), -1.0)
    for s in np.nonzero(d["perm_src"] >= 0)[0]:
        a = int(d["perm_src"][s])
        rows[s] = (rank, a // k, a % k, idx.reshape(-1)[a])
    return rows


CASES = [
    dict(R=2, E=8, k=2, N=37, rank_map=0, cf=0.0),
    dict(R=2, E=8, k=3, N=50, rank_map=1, cf=0.9),
    dict(R=4, E=16, k=4, N=23, rank_map=0, cf=0.0),
    dict(R=3, E=10, k=2, N=41, rank_map=1, cf=1.1),
    dict(R=1, E=6, k=2, N=19, rank_map=0, cf=0.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"R{c['R']}E{c['E']}map{c['rank_map']}")
def test_plan_matches_dispatch_tables(case):
    R, E, k, N, rm, cf = case["R"], case["E"], case["k"], case["N"], case["rank_map"], case["cf"]
    tabs = [_tables(r, N, E, k, R, rm, cf, 5)[1] for r in range(R)]
    kept = np.stack([t["kept_counts"] for t in tabs])
    plans = [ep.ExchangePlan(kept, E, R, rm, me) for me in range(R)]
    for me, (plan, t) in enumerate(zip(plans, tabs)):
        # send chunks are the dispatch's expert segments, in send order, tiling the kept rows
        assert plan.send_rows == t["num_kept"] == kept[me].sum()
        off = 0
        for (dst, e, o, n) in plan.send_chunks:
            assert o == off and o == t["expert_start"][e] and n == t["kept_counts"][e]
            assert e in ep.experts_of_rank(dst, E, R, rm)
            off += n
        for dst in range(R):    # one rank's chunks are its rank segment of the send buffer
            rows = sum(n for (r, _, _, n) in plan.send_chunks if r == dst)
            assert rows == t["rank_counts"][dst]
        # receive side: expert-major, contiguous, every source's chunk sized as sent
        off = 0
        for i, e in enumerate(plan.local_experts):
            assert plan.local_start[i] == off
            assert plan.local_kept[i] == kept[:, e].sum()
            for src in range(R):
                (s2, e2, o, n) = plan.recv_chunks[i * R + src]
                assert (s2, e2, o) == (src, e, off) and n == kept[src, e]
                assert plans[src].send_offset(me, e)[1] == n
                off += n
        assert plan.recv_rows == off
    # every expert has exactly one owner
    owners = sorted(e for p in plans for e in p.local_experts)
    assert owners == list(range(E))


def test_loopback_exchange_round_trip():
    """All ranks in one process: rows reach their experts' owners and come back."""
    R, E, k, N, rm, cf = 3, 12, 3, 29, 1, 1.2
    tabs = [_tables(r, N, E, k, R, rm, cf, 9) for r in range(R)]
    kept = np.stack([t[1]["kept_counts"] for t in tabs])
    plans = [ep.ExchangePlan(kept, E, R, rm, me) for me in range(R)]
    send = [torch.from_numpy(_send_rows(r, *tabs[r], k)) for r in range(R)]
    recv = [torch.full((max(p.recv_rows, 1), 4), -7.0, dtype=torch.float64) for p in plans]
    ep.exchange_loopback(plans, send, recv)
    for me, p in enumerate(plans):
        _check_received(me, p, recv[me], tabs, k)
    back = [torch.full_like(s, -5.0) for s in send]
    res = [r.clone() for r in recv]
    for r in res:
        r[:, 3] += 1000.0
    ep.exchange_loopback(plans, back, res, reverse=True)
    for r in range(R):
        kept_rows = np.nonzero(tabs[r][1]["perm_src"] >= 0)[0]
        want = send[r][kept_rows].clone()
        want[:, 3] += 1000.0
        assert torch.equal(back[r][kept_rows], want)


def _scales(rows):
    """A second, 1-D buffer aligned with the rows (as INT8 scales are with codes)."""
    return (rows[:, 0] * 1000 + rows[:, 1]).to(torch.float32).contiguous()


def test_loopback_exchange_of_row_aligned_pairs():
    """A payload of two row-aligned tensors (codes + scales) moves chunk by chunk together."""
    R, E, k, N, rm, cf = 2, 8, 2, 33, 0, 0.0
    tabs = [_tables(r, N, E, k, R, rm, cf, 21) for r in range(R)]
    kept = np.stack([t[1]["kept_counts"] for t in tabs])
    plans = [ep.ExchangePlan(kept, E, R, rm, me) for me in range(R)]
    send = [torch.from_numpy(_send_rows(r, *tabs[r], k)) for r in range(R)]
    pairs = [(s_, _scales(s_)) for s_ in send]
    recv = [(torch.full((max(p.recv_rows, 1), 4), -7.0, dtype=torch.float64),
             torch.full((max(p.recv_rows, 1),), -7.0)) for p in plans]
    ep.exchange_loopback(plans, pairs, recv)
    for me, p in enumerate(plans):
        _check_received(me, p, recv[me][0], tabs, k)
        rows = p.recv_rows
        assert torch.equal(recv[me][1][:rows], _scales(recv[me][0][:rows]))


def _check_received(me, plan, recv, tabs, k):
    for (src, e, off, n) in plan.recv_chunks:
        idx, d = tabs[src]
        st = d["expert_start"][e]
        exp = np.array([(src, a // k, a % k, e) for a in d["perm_src"][st:st + n]], np.float64)
        got = recv[off:off + n].numpy()
        if n:
            np.testing.assert_array_equal(got, exp.reshape(n, 4))
            assert np.all(np.diff(got[:, 1]) > 0)       # each source's rows in token order


def _worker(rank, world, port, case, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        R, E, k, N, rm, cf = world, case["E"], case["k"], case["N"], case["rank_map"], case["cf"]
        tabs = [_tables(r, N, E, k, R, rm, cf, 3) for r in range(R)]
        idx, d = tabs[rank]
        kept = ep.gather_kept(torch.from_numpy(d["kept_counts"].astype(np.int32)))
        plan = ep.ExchangePlan(kept, E, R, rm, rank)
        send = torch.from_numpy(_send_rows(rank, idx, d, k))
        recv = torch.full((max(plan.recv_rows, 1), 4), -7.0, dtype=torch.float64)
        ep.exchange_dist(plan, send, recv)
        _check_received(rank, plan, recv, tabs, k)
        # a row-aligned pair (as INT8 codes + scales) takes the same path
        recv2 = (torch.full_like(recv, -3.0), torch.full((recv.shape[0],), -3.0))
        ep.exchange_dist(plan, (send, _scales(send)), recv2)
        assert torch.equal(recv2[0][:plan.recv_rows], recv[:plan.recv_rows])
        assert torch.equal(recv2[1][:plan.recv_rows], _scales(recv[:plan.recv_rows]))
        res = recv.clone()
        res[:, 3] += 1000.0                              # the "expert" marks its result
        back = torch.full_like(send, -5.0)
        ep.exchange_dist(plan, back, res, reverse=True)
        kept_rows = np.nonzero(d["perm_src"] >= 0)[0]
        want = send[kept_rows].clone()
        want[:, 3] += 1000.0
        assert torch.equal(back[kept_rows], want)
        q.put((rank, "ok", plan.recv_rows))
    except Exception as exc:                             # report, do not hang the peer
        q.put((rank, repr(exc), -1))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [dict(E=8, k=2, N=37, rank_map=0, cf=0.0),
                                  dict(E=10, k=3, N=45, rank_map=1, cf=0.8)],
                         ids=["contiguous", "round_robin_capacity"])
def test_exchange_gloo_two_ranks(case):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 31500 + (os.getpid() % 2000) + case["E"]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, case, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert [r[1] for r in res] == ["ok", "ok"], res
    assert all(p.exitcode == 0 for p in procs)


def test_receive_capacity_check_is_the_same_on_every_rank():
    """A plan that would overflow one rank's receive buffers is refused by every rank
    (each rank checks all ranks' plans against the shared capacity)."""
    R, E = 2, 8
    kept = np.zeros((R, E), np.int64)
    kept[:, 0] = 50                     # both ranks send 50 rows to expert 0 (rank 0)
    plans = [ep.ExchangePlan(kept, E, R, 0, me) for me in range(R)]
    assert [p.recv_rows for p in plans] == [100, 0]

    class Stub:                          # RankLayer.check_plan without device buffers
        recv_capacity, rank = 64, 1
        check_plan = ep.RankLayer.check_plan
    with pytest.raises(ValueError, match="would receive 100 rows"):
        for other in range(R):
            Stub().check_plan(plans[other])


# ---------------------------------------------------------------- source groups, overlap

@pytest.mark.parametrize("R,G", [(2, 2), (4, 2), (4, 4), (3, 2), (5, 3)])
def test_source_groups_cover_every_distance_once(R, G):
    groups = ep.source_groups(R, G)
    assert len(groups) == min(G, R)
    assert sorted(j for g in groups for j in g) == list(range(R))
    assert groups[0][0] == 0                    # a rank's own rows come first
    assert all(g for g in groups)


@pytest.mark.parametrize("case", CASES[:4], ids=lambda c: f"R{c['R']}E{c['E']}map{c['rank_map']}")
@pytest.mark.parametrize("G", [2, 4])
def test_grouped_plan_layout(case, G):
    """Group-major receive layout: the same chunks as the plain plan, each source group
    one block whose expert segments are contiguous, and both ends of every chunk agree
    on the step that moves it."""
    R, E, k, N, rm, cf = case["R"], case["E"], case["k"], case["N"], case["rank_map"], case["cf"]
    tabs = [_tables(r, N, E, k, R, rm, cf, 7)[1] for r in range(R)]
    kept = np.stack([t["kept_counts"] for t in tabs])
    plain = [ep.ExchangePlan(kept, E, R, rm, me) for me in range(R)]
    plans = [ep.ExchangePlan(kept, E, R, rm, me, groups=G) for me in range(R)]
    for me, (p, q) in enumerate(zip(plans, plain)):
        assert p.send_chunks == q.send_chunks and p.recv_rows == q.recv_rows
        assert sorted((s, e, n) for (s, e, _, n) in p.recv_chunks) == \
            sorted((s, e, n) for (s, e, _, n) in q.recv_chunks)
        g_prev = 0
        for g in range(p.G):
            g0, g1 = p.group_rows[g]
            assert g0 == g_prev
            g_prev = g1
            srcs = p.group_sources[g]
            assert srcs == sorted((me - j) % R for j in p.dist_groups[g])
            for i, e in enumerate(p.local_experts):
                start, n = p.group_start[g][i], p.group_kept[g][i]
                assert n == sum(kept[s, e] for s in srcs)
                chunks = [(s, off, m) for (s, ee, off, m), st in zip(p.recv_chunks, p.recv_step)
                          if ee == e and st == g]
                assert [c[0] for c in chunks] == srcs     # sources ascending in a segment
                off = g0 + start
                for (s, o, m) in chunks:
                    assert o == off
                    off += m
                assert off == g0 + start + n
        assert g_prev == p.recv_rows
        # the step that sends a chunk at its source is the step that receives it here
        for (dst, e, _, n), st in zip(p.send_chunks, p.send_step):
            other = plans[dst]
            (j,) = [i for i, c in enumerate(other.recv_chunks) if c[0] == me and c[1] == e]
            assert other.recv_step[j] == st


@pytest.mark.parametrize("R,E,rm,G", [(2, 8, 0, 2), (4, 16, 1, 2), (3, 9, 1, 3)])
def test_static_plan_is_the_padded_dispatch_layout(R, E, rm, G):
    """With the capacity-padded send buffer the chunks are whole expert blocks of C rows
    at the dispatch's expert_start: the plan needs no counts."""
    k, N, cf = 2, 40, 1.0
    for me in range(R):
        idx = _routing(me, N, E, k, 3)
        d = oracle.dispatch(idx, E, R, rm, cf, mode=1)
        C = d["send_rows"] // E
        p = ep.StaticExchangePlan(E, R, rm, me, C, groups=G)
        assert p.send_rows == d["send_rows"]
        for (dst, e, off, n) in p.send_chunks:
            assert n == C and off == d["expert_start"][e]
            assert e in ep.experts_of_rank(dst, E, R, rm)
            # every kept row of the block lies in the chunk
            assert d["kept_counts"][e] <= C
        assert p.recv_rows == R * C * len(p.local_experts)
        for g in range(p.G):
            assert p.group_kept[g] == [C * len(p.group_sources[g])] * len(p.local_experts)


def _overlap_worker(rank, world, port, case, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        R, E, k, N, rm, cf, G = world, case["E"], case["k"], case["N"], case["rank_map"], \
            case["cf"], case["G"]
        static = case.get("static", False)
        tabs = [_tables(r, N, E, k, R, rm, cf, 11) for r in range(R)]
        idx, d = tabs[rank]
        if static:
            idx_ = idx
            d = oracle.dispatch(idx_, E, R, rm, cf, mode=1)
            plan = ep.StaticExchangePlan(E, R, rm, rank, d["send_rows"] // E, groups=G)
        else:
            kept = ep.gather_kept(torch.from_numpy(d["kept_counts"].astype(np.int32)))
            plan = ep.ExchangePlan(kept, E, R, rm, rank, groups=G)
        send = torch.from_numpy(_send_rows(rank, idx, d, k))
        recv = torch.full((max(plan.recv_rows, 1), 4), -7.0, dtype=torch.float64)
        res = torch.full_like(recv, -9.0)
        back = torch.full_like(send, -5.0)
        done = []

        def compute(g):                  # the "experts" of group g mark their rows
            g0, g1 = plan.group_rows[g]
            res[g0:g1] = recv[g0:g1]
            res[g0:g1, 3] += 1000.0 * (g + 1)
            done.append(g)
        works = ep.overlapped_exchange(plan, send, recv, back, res, compute)
        for wk in works:
            wk.wait()
        assert done == list(range(plan.G))
        kept_rows = np.nonzero(d["perm_src"] >= 0)[0]
        want = send[kept_rows].clone()
        # each kept row came back from the group that holds its source (this rank) at
        # the receiver, marked by that group
        dst_of = {e: dst for dst in range(R) for e in ep.experts_of_rank(dst, E, R, rm)}
        for i, s_row in enumerate(kept_rows):
            e = int(send[s_row, 3])
            j = (rank - dst_of[e]) % R            # my distance from the expert's owner
            g = [gi for gi, js in enumerate(ep.source_groups(R, G)) if j in js][0]
            want[i, 3] += 1000.0 * (g + 1)
        assert torch.equal(back[kept_rows], want)
        q.put((rank, "ok", plan.recv_rows))
    except Exception as exc:                             # report, do not hang the peer
        q.put((rank, repr(exc), -1))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [dict(E=8, k=2, N=37, rank_map=0, cf=0.0, G=2),
                                  dict(E=10, k=3, N=45, rank_map=1, cf=0.8, G=2),
                                  dict(E=8, k=2, N=30, rank_map=0, cf=1.0, G=2, static=True)],
                         ids=["contiguous", "round_robin_capacity", "static_padded"])
def test_overlapped_exchange_gloo_two_ranks(case):
    """The overlapped schedule of run_layer_dist (overlapped_exchange) between two gloo
    ranks: group by group the rows reach the experts' owner, the owner's per-group
    computation sees exactly that group's rows, and every result returns to its row."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 33500 + (os.getpid() % 2000) + case["E"] + 7 * case["k"] + (50 if case.get("static") else 0)
    procs = [ctx.Process(target=_overlap_worker, args=(r, 2, port, case, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert [r[1] for r in res] == ["ok", "ok"], res
    assert all(p.exitcode == 0 for p in procs)
