"""The rank-local zigzag ring driver with the library's kernels, its P ranks
run in one process on one GPU through the loopback transport: every rank
computes on its own chunk pair and on K/V pairs received into local staging
buffers, and its dK/dV come back to it through the ring. The result must
equal monolithic attention (GPU) and the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import long_context_causal_blockwise_gb300 as lcb
from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo
from long_context_causal_blockwise_gb300.ring import LoopbackRing, RingRank
from parity import assert_bf16_close, assert_lse_close, to64

pytestmark = pytest.mark.gpu
D = 128


@pytest.mark.parametrize("S,H,P,fused", [(4096, 2, 4, True), (3072, 2, 3, True), (1200, 2, 3, False),
                                         (2048, 3, 1, True), (2048, 2, 4, False)])
def test_loopback_ring_vs_monolithic_and_oracle(S, H, P, fused):
    q, k, v, do = gaussian_qkvdo(1, H, S, D, seed=S + P)
    perm, _ = lcb.zigzag_schedule(S, P)
    perm_t = torch.as_tensor(perm, device="cuda", dtype=torch.long)
    c2 = S // P
    # each rank's chunk pair, copied out of the global tensors (its own memory)
    local = lambda x, r: x[:, perm_t[r * c2:(r + 1) * c2]].contiguous()  # noqa: E731
    hub = LoopbackRing(P)
    ranks = [RingRank(r, P, S, hub.transport(r)) for r in range(P)]
    mine = [[local(x, r) for x in (q, k, v, do)] for r in range(P)]
    fwd = hub.run([rk.forward_steps(*mine[r][:3]) for r, rk in enumerate(ranks)])
    bwd = hub.run([rk.backward_steps(*mine[r][:3], fwd[r][0], fwd[r][1], mine[r][3], fused=fused)
                   for r, rk in enumerate(ranks)])
    o, lse = lcb.attn_fwd(q, k, v)
    dq, dk, dv = lcb.attn_bwd(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    cat = lambda xs, dim=1: torch.cat(xs, dim=dim)  # noqa: E731  (rank order = zigzag order)
    oz, lsez = cat([f[0] for f in fwd]), cat([f[1] for f in fwd], 2)
    dqz, dkz, dvz = (cat([b[i] for b in bwd]) for i in range(3))
    assert_bf16_close(to64(oz), to64(o[:, perm_t]), "O ring vs monolithic")
    assert_lse_close(to64(lsez), to64(lse[:, :, perm_t]))
    for name, got, ref in (("dQ", dqz, dq), ("dK", dkz, dk), ("dV", dvz, dv)):
        assert_bf16_close(to64(got), to64(ref[:, perm_t]), f"{name} ring vs monolithic")
    want = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), True, D ** -0.5)
    inv = np.argsort(np.asarray(perm))
    assert_bf16_close(to64(oz)[:, inv], want["o"], "O ring vs oracle")
    assert_lse_close(to64(lsez)[:, :, inv], want["lse"])
    for name, got in (("dq", dqz), ("dk", dkz), ("dv", dvz)):
        assert_bf16_close(to64(got)[:, inv], want[name], f"{name} ring vs oracle")


def test_loopback_ring_equals_one_device_emulation():
    """The ring driver and the one-device emulation (grouped launches over the
    zigzag-ordered tensors) run the same tasks: O and LSE bit for bit, dK and
    dV bit for bit (fp32 sums in the same step order), dQ within rounding."""
    S, H, P = 4096, 2, 4
    q, k, v, do = gaussian_qkvdo(1, H, S, D, seed=99)
    plan = lcb.zigzag.ZigzagPlan(S, P, "cuda")
    qz, kz, vz, doz = (plan.gather(x) for x in (q, k, v, do))
    oz, lsez, _ = lcb.zigzag_attention_fwd(qz, kz, vz, plan)
    gz = lcb.zigzag_attention_bwd(qz, kz, vz, oz, lsez, doz, plan)
    c2 = S // P
    hub = LoopbackRing(P)
    ranks = [RingRank(r, P, S, hub.transport(r)) for r in range(P)]
    part = lambda x, r: x[:, r * c2:(r + 1) * c2].contiguous()  # noqa: E731
    fwd = hub.run([rk.forward_steps(part(qz, r), part(kz, r), part(vz, r)) for r, rk in enumerate(ranks)])
    bwd = hub.run([rk.backward_steps(part(qz, r), part(kz, r), part(vz, r), fwd[r][0], fwd[r][1], part(doz, r))
                   for r, rk in enumerate(ranks)])
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([f[0] for f in fwd], 1), oz)
    assert torch.equal(torch.cat([f[1] for f in fwd], 2), lsez)
    assert torch.equal(torch.cat([b[1] for b in bwd], 1), gz[1])
    assert torch.equal(torch.cat([b[2] for b in bwd], 1), gz[2])
    dq = torch.cat([b[0] for b in bwd], 1).float()
    assert (dq - gz[0].float()).abs().max().item() <= 2 ** -7 * gz[0].float().abs().max().item()


def test_loopback_ring_config3_131072_p8():
    """B=1, H=32, S=131072 over P=8 ranks (C3's shape) through the rank-local
    driver: O, LSE, dK and dV bit for bit those of the one-device emulation,
    dQ within rounding, and O, LSE, dQ against the oracle on sampled rows plus
    every chunk edge of every head."""
    from long_context_causal_blockwise_gb300.inputs import sample_rows
    from parity import oracle_rows_by_head, rows_budget

    S, H, P = 131072, 32, 8
    q, k, v, do = gaussian_qkvdo(1, H, S, D, seed=0)
    plan = lcb.zigzag.ZigzagPlan(S, P, "cuda")
    qz, kz, vz, doz = (plan.gather(x) for x in (q, k, v, do))
    del q, k, v, do
    oz, lsez, _ = lcb.zigzag_attention_fwd(qz, kz, vz, plan)
    gz = lcb.zigzag_attention_bwd(qz, kz, vz, oz, lsez, doz, plan)
    c2 = S // P
    hub = LoopbackRing(P)
    ranks = [RingRank(r, P, S, hub.transport(r)) for r in range(P)]
    part = lambda x, r: x[:, r * c2:(r + 1) * c2].contiguous()  # noqa: E731
    mine = [[part(x, r) for x in (qz, kz, vz, doz)] for r in range(P)]
    fwd = hub.run([rk.forward_steps(*mine[r][:3]) for r, rk in enumerate(ranks)])
    bwd = hub.run([rk.backward_steps(*mine[r][:3], fwd[r][0], fwd[r][1], mine[r][3]) for r, rk in enumerate(ranks)])
    torch.cuda.synchronize()
    o_r = torch.cat([f[0] for f in fwd], 1)
    lse_r = torch.cat([f[1] for f in fwd], 2)
    dq_r, dk_r, dv_r = (torch.cat([b_[i] for b_ in bwd], 1) for i in range(3))
    del fwd, bwd, mine
    assert torch.equal(o_r, oz) and torch.equal(lse_r, lsez)
    assert torch.equal(dk_r, gz[1]) and torch.equal(dv_r, gz[2])
    assert (dq_r.float() - gz[0].float()).abs().max().item() <= 2 ** -7 * gz[0].float().abs().max().item()
    # against the oracle in natural order
    inv = np.argsort(np.asarray(plan.perm))
    inv_t = torch.as_tensor(inv, device="cuda")
    q, k, v, do = (plan.scatter(x) for x in (qz, kz, vz, doz))
    rows = sample_rows(S, rows_budget(1024), seed=5)
    c = S // (2 * P)
    rows = np.unique(np.concatenate([rows, [e for j in range(1, 2 * P) for e in (j * c - 1, j * c)]]))
    refs = oracle_rows_by_head(q, k, v, do, rows, True, D ** -0.5)
    zpos = inv_t[torch.as_tensor(rows, device="cuda")]
    assert_bf16_close(to64(o_r[:, zpos]), np.concatenate([x["o"] for x in refs], 2), "O ring C3 vs oracle")
    assert_lse_close(to64(lse_r[:, :, zpos]), np.concatenate([x["lse"] for x in refs], 1))
    assert_bf16_close(to64(dq_r[:, zpos]), np.concatenate([x["dq"] for x in refs], 2), "dQ ring C3 vs oracle")


@pytest.mark.parametrize("S,H,P,fused", [(4096, 2, 4, True), (1200, 2, 3, False), (2048, 2, 1, True)])
def test_loopback_contiguous_ring_vs_monolithic_and_oracle(S, H, P, fused):
    """The plain ring (rank r holds rows [r S/P, (r+1) S/P)) through the same driver."""
    q, k, v, do = gaussian_qkvdo(1, H, S, D, seed=S + 7 * P)
    n = S // P
    hub = LoopbackRing(P, time_ranks=True)
    ranks = [RingRank(r, P, S, hub.transport(r), schedule="contiguous") for r in range(P)]
    mine = [[x[:, r * n:(r + 1) * n].contiguous() for x in (q, k, v, do)] for r in range(P)]
    fwd = hub.run([rk.forward_steps(*mine[r][:3]) for r, rk in enumerate(ranks)])
    bwd = hub.run([rk.backward_steps(*mine[r][:3], fwd[r][0], fwd[r][1], mine[r][3], fused=fused)
                   for r, rk in enumerate(ranks)])
    per_rank = hub.rank_ms()
    o = torch.cat([f[0] for f in fwd], 1)
    lse = torch.cat([f[1] for f in fwd], 2)
    dq, dk, dv = (torch.cat([b_[i] for b_ in bwd], 1) for i in range(3))
    torch.cuda.synchronize()
    want = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), True, D ** -0.5)
    assert_bf16_close(to64(o), want["o"], "O plain ring vs oracle")
    assert_lse_close(to64(lse), want["lse"])
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_bf16_close(to64(got), want[name], f"{name} plain ring vs oracle")
    assert len(per_rank) == P and all(t > 0 for t in per_rank)
