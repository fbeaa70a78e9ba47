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
