"""Zigzag ring attention across ranks: the rank-local driver.

Ring attention over sequence shards ("EasyContext核心技术解析：序列并行与Flash
Attention的完美结合", §1 "序列并行技术"; compute and communication overlapped,
same page, 技术实现细节 › 异步通信优化) with the zigzag split
("EasyContext代码解析200行核心训练脚本实现原理", §模型并行策略解析
zigzag_ring_attn): rank r of P holds sequence chunks r and 2P-1-r of Q, K,
V (its 2c rows, c = S / 2P) and never sees another rank's memory.

The plain (contiguous) ring is the same driver with schedule="contiguous":
rank r holds rows [r S/P, (r+1) S/P), and its steps that hold a later
rank's keys compute nothing.

Forward, ring step s = 0 .. P-1: the rank holds the K/V pair of rank
src = (r - s) mod P in a local buffer. Before computing with it, it starts
sending that pair to rank r+1 and receiving rank r-1's pair into a second
local staging buffer, so the transfer runs while the step computes. The
step's task (DIAG, LOWER or UPPER, from zigzag_schedule) runs as one
attn_fwd_ex call on local memory: step 0 stores the rank's fp32 (O, LSE)
accumulator, later steps merge into it in the kernel epilogue.

Backward: every task uses the rank's final LSE and Delta. dQ stays on the
rank. The fp32 dK/dV accumulators of the keys a rank holds travel with those
keys: at step s the rank adds its contribution to the accumulators that
arrived with src's K/V, then passes K, V and the accumulators on. After step
P-1 one more hop returns the accumulators to their owner, which casts them to
bf16.

Transports (`exchange(send, recv)` starts the transfers and returns a handle
whose wait() completes them):
  DistRingTransport  torch.distributed point-to-point to r+1 / from r-1
                     (gloo between CPU processes, NCCL between GPUs);
  LoopbackRing       the P ranks of one process on one device, transfers
                     as device copies (ranks stepped round-robin).
Every piece of arithmetic runs in libattn.so kernels (RingCompute); only the
transfers are the transport's.
"""

import torch

from . import _lib


class _Done:
    def wait(self):
        return None


class _Requests:
    def __init__(self, reqs):
        self.reqs = reqs

    def wait(self):
        for r in self.reqs:
            r.wait()


class DistRingTransport:
    """Point-to-point over a torch.distributed process group: this rank sends
    to rank+1 and receives from rank-1 (ring order = group rank order)."""

    def __init__(self, group=None):
        import torch.distributed as dist

        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        to_global = (lambda r: dist.get_global_rank(group, r)) if group is not None else (lambda r: r)
        self.next = to_global((self.rank + 1) % self.world)
        self.prev = to_global((self.rank - 1) % self.world)

    def exchange(self, send, recv):
        if self.world == 1:
            for d, s in zip(recv, send):
                d.copy_(s)
            return _Done()
        dist = self.dist
        ops = [dist.P2POp(dist.isend, t, self.next, self.group) for t in send]
        ops += [dist.P2POp(dist.irecv, t, self.prev, self.group) for t in recv]
        return _Requests(dist.batch_isend_irecv(ops))


class RingCompute:
    """The library calls one ring step makes on a rank's local tensors."""

    def fwd(self, task, q, k, v, o_acc, lse, scale):
        qs = slice(task["q_rel"], task["q_rel"] + task["q_len"])
        ks = slice(task["k_rel"], task["k_rel"] + task["k_len"])
        _lib.attn_fwd_ex(q[:, qs], k[:, ks], v[:, ks], o_acc[:, qs], lse[:, :, qs], bool(task["causal"]), scale,
                         merge=task["step"] > 0)

    def finish_fwd(self, o_acc, o):
        _lib.cast_f32_bf16(o_acc, o)

    def delta(self, o, do, delta):
        _lib.attn_bwd_preprocess(o, do, delta)

    def bwd(self, task, q, k, v, lse, delta, do, dq_acc, dk_acc, dv_acc, scale):
        """Adds the task's dQ into dq_acc (a tiled accumulator when fused) and
        its dK/dV into the travelling accumulators (stored at step 0)."""
        acc = task["step"] > 0
        if dq_acc.dim() == 4 and dq_acc.shape[-1] == 128 * 128:  # tiled: one-pass backward
            t = (task["q_rel"], task["q_len"], task["k_rel"], task["k_len"], task["causal"])
            _lib.attn_bwd_group(q, k, v, lse, delta, do, dq_acc, dk_acc, dv_acc, [t], scale, accumulate=acc)
        else:
            qs = slice(task["q_rel"], task["q_rel"] + task["q_len"])
            ks = slice(task["k_rel"], task["k_rel"] + task["k_len"])
            _lib.attn_bwd_ex(q[:, qs], k[:, ks], v[:, ks], lse[:, :, qs], delta[:, :, qs], do[:, qs], dq_acc[:, qs],
                             dk_acc[:, ks], dv_acc[:, ks], bool(task["causal"]), scale, accumulate=acc)

    def finish_bwd(self, dq_acc, dk_acc, dv_acc, dq, dk, dv):
        if dq_acc.dim() == 4 and dq_acc.shape[-1] == 128 * 128:
            _lib.dq_untile(dq_acc, dq)
        else:
            _lib.cast_f32_bf16(dq_acc, dq)
        _lib.cast_f32_bf16(dk_acc, dk)
        _lib.cast_f32_bf16(dv_acc, dv)


def rank_tasks(S, P, rank, schedule="zigzag"):
    """Rank `rank`'s ring tasks in step order, with row offsets relative to
    its own rows (q_rel) and to the holder's rows (k_rel). schedule "zigzag"
    (chunks r and 2P-1-r) or "contiguous" (the plain ring, rows [r S/P, (r+1)
    S/P)); either way a rank holds S/P rows."""
    sched = {"zigzag": _lib.zigzag_schedule, "contiguous": _lib.ring_schedule}[schedule]
    _, tasks = sched(S, P)
    n = S // P
    mine = sorted((t for t in tasks if t["rank"] == rank), key=lambda t: t["step"])
    for t in mine:
        t["q_rel"] = t["q_off"] - rank * n
        t["k_rel"] = t["k_off"] - t["src"] * n
    return mine


class RingRank:
    """One rank of the ring: its own rows, its tasks, a transport.

    schedule "zigzag" balances the causal work across ranks; "contiguous" is
    the plain ring (rank r's work grows with r; its steps that hold a later
    rank's keys have nothing to compute and only pass the keys on)."""

    def __init__(self, rank, P, S, transport, compute=None, scale=None, schedule="zigzag"):
        if schedule == "zigzag" and S % (2 * P):
            raise ValueError("the zigzag split needs S a multiple of 2P")
        if S % P:
            raise ValueError("the ring needs S a multiple of P")
        self.rank, self.P, self.S = rank, P, S
        self.n = S // P  # rows per rank
        self.schedule = schedule
        self.tasks = rank_tasks(S, P, rank, schedule)
        self.transport = transport
        self.compute = RingCompute() if compute is None else compute
        self.scale = scale

    def forward_steps(self, q, k, v):
        """Generator of the forward. It yields once per ring step, the list of
        transfer handles that step started (the caller waits on them before
        resuming it), and returns (o bf16, lse fp32 [1, H, 2c], o_acc fp32) of
        this rank's rows."""
        B, n, H, D = q.shape
        if B != 1 or n != self.n:
            raise ValueError("a rank holds [1, S/P, H, D] of each tensor")
        scale = D ** -0.5 if self.scale is None else self.scale
        o_acc = torch.empty((1, n, H, D), dtype=torch.float32, device=q.device)
        lse = torch.empty((1, H, n), dtype=torch.float32, device=q.device)
        stage = [(torch.empty_like(k), torch.empty_like(v)) for _ in range(2 if self.P > 1 else 0)]
        cur = (k, v)
        for s, task in enumerate(self.tasks):
            handles = []
            if s + 1 < self.P:  # pass the pair on while this step computes with it
                nxt = stage[s % 2]
                handles.append(self.transport.exchange(list(cur), list(nxt)))
            if task["q_len"] and task["k_len"]:
                self.compute.fwd(task, q, cur[0], cur[1], o_acc, lse, scale)
            yield handles
            if s + 1 < self.P:
                cur = nxt
        o = torch.empty_like(q)
        self.compute.finish_fwd(o_acc, o)
        return o, lse, o_acc

    def backward_steps(self, q, k, v, o, lse, do, fused=True):
        """Generator of the backward (same protocol); returns (dq, dk, dv) bf16
        of this rank's rows, dK/dV complete once the last hop has arrived."""
        B, n, H, D = q.shape
        scale = D ** -0.5 if self.scale is None else self.scale
        dev = q.device
        delta = torch.empty((1, H, n), dtype=torch.float32, device=dev)
        self.compute.delta(o, do, delta)
        # the tiled dQ accumulator takes query blocks that start on 128-row tiles
        fused = fused and all(t["q_rel"] % 128 == 0 for t in self.tasks)
        # dQ: the one-pass backward adds into a zeroed tiled accumulator; the
        # two-pass form stores at step 0 (the DIAG task covers every local row)
        dq_acc = (_lib.dq_tiles_zeros(1, H, n, dev) if fused else
                  torch.empty((1, n, H, D), dtype=torch.float32, device=dev))
        f32 = lambda: torch.empty((1, n, H, D), dtype=torch.float32, device=dev)  # noqa: E731
        acc = (f32(), f32())  # accumulators of the keys held at step 0 (this rank's own), stored at step 0
        kv_stage = [(torch.empty_like(k), torch.empty_like(v)) for _ in range(2 if self.P > 1 else 0)]
        acc_stage = [(f32(), f32()) for _ in range(2)]
        cur = (k, v)
        for s, task in enumerate(self.tasks):
            handles = []
            if s + 1 < self.P:  # K and V are read-only: pass them on before computing
                nxt = kv_stage[s % 2]
                handles.append(self.transport.exchange(list(cur), list(nxt)))
            if task["q_len"] and task["k_len"]:
                self.compute.bwd(task, q, cur[0], cur[1], lse, delta, do, dq_acc, acc[0], acc[1], scale)
            # the accumulators go on with this step's contribution; the hop after
            # step P-1 brings every rank its own keys' accumulators
            nacc = acc_stage[s % 2]
            handles.append(self.transport.exchange(list(acc), list(nacc)))
            yield handles
            acc = nacc
            if s + 1 < self.P:
                cur = nxt
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        self.compute.finish_bwd(dq_acc, acc[0], acc[1], dq, dk, dv)
        return dq, dk, dv


def run_rank(gen):
    """Drives one rank's generator to completion across processes: every
    handle a step started is waited on before the next step."""
    while True:
        try:
            handles = next(gen)
        except StopIteration as stop:
            return stop.value
        for h in handles:
            h.wait()


class _Ticket:
    def wait(self):
        return None


class LoopbackRing:
    """P ranks in one process on one device. Every rank makes the same
    sequence of exchange() calls; the k-th exchange of rank r sends to the
    k-th of rank r+1. The ranks are stepped round-robin, one ring step each,
    and after each round every posted transfer is made as a device copy on
    the current stream: after the senders' step, before the receivers' next."""

    def __init__(self, P, time_ranks=False):
        self.P = P
        self.posted = [[] for _ in range(P)]
        # optional: CUDA events around every rank's steps (its kernels only, not the transfers)
        self.events = [[] for _ in range(P)] if time_ranks else None

    def rank_ms(self):
        """Milliseconds of kernel time per rank (time_ranks=True; synchronises)."""
        torch.cuda.synchronize()
        return [sum(a.elapsed_time(b) for a, b in evs) for evs in self.events]

    def transport(self, rank):
        hub = self

        class _T:
            def exchange(self, send, recv):
                hub.posted[rank].append((send, recv))
                return _Ticket()

        return _T()

    def _deliver(self):
        n = len(self.posted[0])
        if any(len(q) != n for q in self.posted):
            raise RuntimeError("ranks posted different numbers of transfers")
        for k in range(n):
            for r in range(self.P):
                send = self.posted[r][k][0]
                recv = self.posted[(r + 1) % self.P][k][1]
                for d, t in zip(recv, send):
                    d.copy_(t)
        self.posted = [[] for _ in range(self.P)]

    def run(self, gens):
        """Steps every rank's generator round-robin; returns their results."""
        if len(gens) != self.P:
            raise ValueError("one generator per rank")
        results = [None] * self.P
        live = list(range(self.P))
        while live:
            still = []
            for r in live:
                if self.events is not None:
                    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    ev[0].record()
                try:
                    next(gens[r])
                    still.append(r)
                except StopIteration as stop:
                    results[r] = stop.value
                if self.events is not None:
                    ev[1].record()
                    self.events[r].append(ev)
            if still and len(still) != self.P:
                raise RuntimeError("ranks left the ring at different steps")
            self._deliver()
            live = still
        return results
