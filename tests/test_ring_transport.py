"""The rank-local zigzag ring driver's transport and ownership logic on the CPU.

A tracing stand-in for the library's kernels records, at every ring step,
whose K/V the rank holds (K is filled with its owner's rank, V with 100 +
rank) and marks the travelling dK/dV accumulators with the contributing
rank and the task kind. The record must match the oracle's zigzag schedule
bit for bit (src, task kind, offsets), and after the backward every rank
must hold its own keys' accumulators carrying exactly one mark from each
rank, of the kind the oracle assigns. Run in one process through the
loopback transport and as real gloo ranks (world size 2 and 4) through
torch.distributed point-to-point."""

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class TraceCompute:
    """Stands in for the kernels: records what each step sees, marks accumulators."""

    def __init__(self, rank):
        self.rank = rank
        self.fwd_seen, self.bwd_seen = [], []

    def fwd(self, task, q, k, v, o_acc, lse, scale):
        self.fwd_seen.append((task["step"], int(k[0, 0, 0, 0]), int(v[0, 0, 0, 0]) - 100,
                              task["kind"], task["q_rel"], task["q_len"], task["k_rel"], task["k_len"], task["causal"]))

    def finish_fwd(self, o_acc, o):
        pass

    def delta(self, o, do, delta):
        pass

    def bwd(self, task, q, k, v, lse, delta, do, dq_acc, dk_acc, dv_acc, scale):
        self.bwd_seen.append((task["step"], int(k[0, 0, 0, 0])))
        if task["step"] == 0:  # the kernels store at step 0
            dk_acc.zero_()
            dv_acc.zero_()
        dk_acc[0, 0, 0, self.rank] += 1.0
        dv_acc[0, 0, 0, self.rank] += 1.0 + task["kind"]

    def finish_bwd(self, dq_acc, dk_acc, dv_acc, dq, dk, dv):
        dk.copy_(dk_acc)
        dv.copy_(dv_acc)


def _local(rank, c, P):
    """Rank `rank`'s chunk pair: K tagged with its owner, V with 100 + owner."""
    shape = (1, 2 * c, 1, max(P, 2))
    q = torch.zeros(shape)
    k = torch.full(shape, float(rank))
    v = torch.full(shape, 100.0 + rank)
    return q, k, v


def _check_rank(rank, P, S, tr, dk, dv):
    _, tasks = oracle.zigzag_schedule(S, P)
    c2 = S // P
    want = sorted((t for t in tasks if t["rank"] == rank), key=lambda t: t["step"])
    assert len(tr.fwd_seen) == P and len(tr.bwd_seen) == P
    for t, f, b in zip(want, tr.fwd_seen, tr.bwd_seen):
        assert f == (t["step"], t["src"], t["src"], t["kind"], t["q_off"] - rank * c2, t["q_len"],
                     t["k_off"] - t["src"] * c2, t["k_len"], t["causal"]), (rank, f, t)
        assert b == (t["step"], t["src"])
    # every rank added exactly one contribution to this rank's keys, of the kind the oracle assigns
    for other in range(P):
        t = next(x for x in tasks if x["rank"] == other and x["src"] == rank)
        assert float(dk[0, 0, 0, other]) == 1.0
        assert float(dv[0, 0, 0, other]) == 1.0 + t["kind"]


@pytest.mark.parametrize("P,c", [(1, 2), (2, 2), (3, 1), (4, 2), (8, 1)])
def test_loopback_ring_routes_kv_and_accumulators(P, c):
    from long_context_causal_blockwise_gb300.ring import LoopbackRing, RingRank

    S = 2 * P * c
    hub = LoopbackRing(P)
    traces = [TraceCompute(r) for r in range(P)]
    ranks = [RingRank(r, P, S, hub.transport(r), compute=traces[r]) for r in range(P)]
    data = [_local(r, c, P) for r in range(P)]
    fwd = hub.run([rk.forward_steps(*data[r]) for r, rk in enumerate(ranks)])
    bwd = hub.run([rk.backward_steps(*data[r], fwd[r][0], fwd[r][1], data[r][0]) for r, rk in enumerate(ranks)])
    for r in range(P):
        _check_rank(r, P, S, traces[r], bwd[r][1], bwd[r][2])
        # the rank's own K/V are untouched by the ring
        assert torch.equal(data[r][1], torch.full_like(data[r][1], float(r)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gloo_rank(rank, world, port, c, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from long_context_causal_blockwise_gb300.ring import DistRingTransport, RingRank, run_rank
    from test_ring_transport import TraceCompute, _check_rank, _local

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        S = 2 * world * c
        tr = TraceCompute(rank)
        rk = RingRank(rank, world, S, DistRingTransport(), compute=tr)
        q, k, v = _local(rank, c, world)
        o, lse, _ = run_rank(rk.forward_steps(q, k, v))
        dq, dk, dv = run_rank(rk.backward_steps(q, k, v, o, lse, q))
        _check_rank(rank, world, S, tr, dk, dv)
        out.put((rank, "ok"))
    except AssertionError as e:  # report, then leave cleanly
        out.put((rank, f"fail: {e}"))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_gloo_ranks_route_kv_and_accumulators(world):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gloo_rank, args=(r, world, port, 2, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(r, "ok") for r in range(world)], got


def test_pins_catch_a_ring_running_backwards():
    """A planted mistake: a transport that delivers to rank r-1 instead of r+1
    (the other ring direction with the schedule's src unchanged) must fail."""
    from long_context_causal_blockwise_gb300.ring import LoopbackRing, RingRank

    class Backwards(LoopbackRing):
        def _deliver(self):
            n = len(self.posted[0])
            for kk in range(n):
                for r in range(self.P):
                    for d, t in zip(self.posted[(r - 1) % self.P][kk][1], self.posted[r][kk][0]):
                        d.copy_(t)
            self.posted = [[] for _ in range(self.P)]

    P, c = 3, 1
    S = 2 * P * c
    hub = Backwards(P)
    traces = [TraceCompute(r) for r in range(P)]
    ranks = [RingRank(r, P, S, hub.transport(r), compute=traces[r]) for r in range(P)]
    data = [_local(r, c, P) for r in range(P)]
    fwd = hub.run([rk.forward_steps(*data[r]) for r, rk in enumerate(ranks)])
    bwd = hub.run([rk.backward_steps(*data[r], fwd[r][0], fwd[r][1], data[r][0]) for r, rk in enumerate(ranks)])
    with pytest.raises(AssertionError):
        for r in range(P):
            _check_rank(r, P, S, traces[r], bwd[r][1], bwd[r][2])


def _check_rank_contiguous(rank, P, S, tr, dk, dv):
    """The plain ring: the steps with work match the oracle's DIAG/FULL tasks,
    and rank `rank`'s keys carry one mark from each rank at or after it."""
    _, tasks = oracle.ring_schedule(S, P)
    n = S // P
    want = sorted((t for t in tasks if t["rank"] == rank and t["kind"] != oracle.TASK_NONE),
                  key=lambda t: t["step"])
    assert len(tr.fwd_seen) == len(want) == rank + 1 and len(tr.bwd_seen) == rank + 1
    for t, f, b in zip(want, tr.fwd_seen, tr.bwd_seen):
        assert f == (t["step"], t["src"], t["src"], t["kind"], t["q_off"] - rank * n, t["q_len"],
                     t["k_off"] - t["src"] * n, t["k_len"], t["causal"]), (rank, f, t)
        assert b == (t["step"], t["src"])
    for other in range(P):
        t = next(x for x in tasks if x["rank"] == other and x["src"] == rank)
        has_work = t["kind"] != oracle.TASK_NONE
        assert float(dk[0, 0, 0, other]) == (1.0 if has_work else 0.0)
        assert float(dv[0, 0, 0, other]) == (1.0 + t["kind"] if has_work else 0.0)


@pytest.mark.parametrize("P,n", [(1, 2), (2, 2), (3, 1), (4, 3), (8, 1)])
def test_loopback_contiguous_ring_routes_kv_and_accumulators(P, n):
    from long_context_causal_blockwise_gb300.ring import LoopbackRing, RingRank

    S = P * n
    hub = LoopbackRing(P)
    traces = [TraceCompute(r) for r in range(P)]
    ranks = [RingRank(r, P, S, hub.transport(r), compute=traces[r], schedule="contiguous") for r in range(P)]
    data = [_local_n(r, n, P) for r in range(P)]
    fwd = hub.run([rk.forward_steps(*data[r]) for r, rk in enumerate(ranks)])
    bwd = hub.run([rk.backward_steps(*data[r], fwd[r][0], fwd[r][1], data[r][0]) for r, rk in enumerate(ranks)])
    for r in range(P):
        _check_rank_contiguous(r, P, S, traces[r], bwd[r][1], bwd[r][2])


def _local_n(rank, n, P):
    shape = (1, n, 1, max(P, 2))
    return torch.zeros(shape), torch.full(shape, float(rank)), torch.full(shape, 100.0 + rank)


def _gloo_rank_contiguous(rank, world, port, n, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from long_context_causal_blockwise_gb300.ring import DistRingTransport, RingRank, run_rank
    from test_ring_transport import TraceCompute, _check_rank_contiguous, _local_n

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        S = world * n
        tr = TraceCompute(rank)
        rk = RingRank(rank, world, S, DistRingTransport(), compute=tr, schedule="contiguous")
        q, k, v = _local_n(rank, n, world)
        o, lse, _ = run_rank(rk.forward_steps(q, k, v))
        dq, dk, dv = run_rank(rk.backward_steps(q, k, v, o, lse, q))
        _check_rank_contiguous(rank, world, S, tr, dk, dv)
        out.put((rank, "ok"))
    except AssertionError as e:
        out.put((rank, f"fail: {e}"))
    finally:
        dist.destroy_process_group()


def test_gloo_ranks_contiguous_ring():
    world = 3
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gloo_rank_contiguous, args=(r, world, port, 2, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(r, "ok") for r in range(world)], got
