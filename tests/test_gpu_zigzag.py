"""Zigzag ring attention emulated on one GPU equals monolithic attention.

The ring's LSE-merged forward and its backward with the final merged
statistics must reproduce monolithic causal attention (GPU, same tolerances)
and the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import long_context_causal_blockwise_gb300 as lcb
from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo, sample_rows
from long_context_causal_blockwise_gb300.zigzag import ZigzagPlan
from parity import assert_bf16_close, assert_lse_close, oracle_rows_by_head, rows_budget, to64

pytestmark = pytest.mark.gpu
D = 128


def _run(S, H, P, seed):
    q, k, v, do = gaussian_qkvdo(1, H, S, D, seed=seed)
    plan = ZigzagPlan(S, P, "cuda")
    qz, kz, vz, doz = (plan.gather(x) for x in (q, k, v, do))
    oz, lsez, _ = lcb.zigzag_attention_fwd(qz, kz, vz, plan)
    dqz, dkz, dvz = lcb.zigzag_attention_bwd(qz, kz, vz, oz, lsez, doz, plan)
    o, lse = lcb.attn_fwd(q, k, v)
    dq, dk, dv = lcb.attn_bwd(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    perm = torch.as_tensor(plan.perm, device="cuda", dtype=torch.long)
    return dict(q=q, k=k, v=v, do=do, plan=plan, perm=perm, oz=oz, lsez=lsez, dqz=dqz, dkz=dkz, dvz=dvz, o=o, lse=lse,
                dq=dq, dk=dk, dv=dv)


def _vs_monolithic(r, tag):
    perm = r["perm"]
    assert_bf16_close(to64(r["oz"]), to64(r["o"][:, perm]), "O zigzag vs monolithic " + tag)
    assert_lse_close(to64(r["lsez"]), to64(r["lse"][:, :, perm]), "LSE zigzag vs monolithic")
    for g in ("dq", "dk", "dv"):
        assert_bf16_close(to64(r[g + "z"]), to64(r[g][:, perm]), f"{g} zigzag vs monolithic " + tag)


@pytest.mark.parametrize("S,H,P", [(2048, 2, 1), (4096, 4, 4), (3072, 2, 3)])
def test_small_zigzag_vs_monolithic_and_oracle(S, H, P):
    r = _run(S, H, P, seed=S + P)
    _vs_monolithic(r, f"S{S} P{P}")
    ref = oracle.attn_bwd(to64(r["q"]), to64(r["k"]), to64(r["v"]), to64(r["do"]), True, D ** -0.5)
    inv = np.argsort(np.asarray(r["plan"].perm))
    assert_bf16_close(to64(r["oz"])[:, inv], ref["o"], "O zigzag vs oracle")
    assert_lse_close(to64(r["lsez"])[:, :, inv], ref["lse"])
    assert_bf16_close(to64(r["dqz"])[:, inv], ref["dq"], "dQ zigzag vs oracle")
    assert_bf16_close(to64(r["dkz"])[:, inv], ref["dk"], "dK zigzag vs oracle")
    assert_bf16_close(to64(r["dvz"])[:, inv], ref["dv"], "dV zigzag vs oracle")


def test_config3_zigzag_131072_p8():
    """B=1, H=32, S=131072, P=8 (16 chunks of 8192): ring result vs monolithic
    on every element, and vs the oracle on 4096 sampled query rows plus every
    chunk edge, on every head."""
    S, H, P = 131072, 32, 8
    r = _run(S, H, P, seed=0)
    _vs_monolithic(r, "C3")
    rows = sample_rows(S, rows_budget(4096), seed=3)
    # every chunk edge of the zigzag split: among the most likely places to go wrong
    c = S // (2 * P)
    edges = [e for j in range(1, 2 * P) for e in (j * c - 1, j * c)]
    rows = np.unique(np.concatenate([rows, edges]))
    refs = oracle_rows_by_head(r["q"], r["k"], r["v"], r["do"], rows, True, D ** -0.5)
    inv = np.argsort(np.asarray(r["plan"].perm))
    zpos = torch.as_tensor(inv[rows], device="cuda")
    assert_bf16_close(to64(r["oz"][:, zpos]), np.concatenate([x["o"] for x in refs], 2), "O C3 sampled vs oracle")
    assert_lse_close(to64(r["lsez"][:, :, zpos]), np.concatenate([x["lse"] for x in refs], 1))
    assert_bf16_close(to64(r["dqz"][:, zpos]), np.concatenate([x["dq"] for x in refs], 2),
                      "dQ C3 sampled vs oracle")


@pytest.mark.parametrize("fused", [True, False])
def test_ring_forward_fused_and_unfused_agree(fused):
    """Both forward step forms (merge in the kernel epilogue, or block result +
    merge kernel) reproduce monolithic attention."""
    S, H, P = 4096, 2, 4
    q, k, v, _ = gaussian_qkvdo(1, H, S, D, seed=77)
    plan = ZigzagPlan(S, P, "cuda")
    qz, kz, vz = (plan.gather(x) for x in (q, k, v))
    oz, lsez, _ = lcb.zigzag_attention_fwd(qz, kz, vz, plan, fused=fused)
    o, lse = lcb.attn_fwd(q, k, v)
    perm = torch.as_tensor(plan.perm, device="cuda", dtype=torch.long)
    assert_bf16_close(to64(oz), to64(o[:, perm]), f"O zigzag fused={fused}")
    assert_lse_close(to64(lsez), to64(lse[:, :, perm]))


@pytest.mark.parametrize("Sq,Sk1,Sk2", [(384, 256, 384), (200, 130, 70)])
def test_forward_merge_mode_vs_oracle(Sq, Sk1, Sk2):
    """attn_fwd_ex in merge mode: the accumulator holds attention over keys
    [0, Sk1); merging the block over keys [Sk1, Sk1 + Sk2) gives attention over
    all keys (oracle, non-causal), and equals the unfused block + merge kernel."""
    H = 3
    g = torch.Generator().manual_seed(Sq + Sk1 + Sk2)
    q, k, v = (torch.randn(1, n, H, D, generator=g).to("cuda", torch.bfloat16) for n in (Sq, Sk1 + Sk2, Sk1 + Sk2))
    scale = D ** -0.5
    k1, v1, k2, v2 = k[:, :Sk1], v[:, :Sk1], k[:, Sk1:], v[:, Sk1:]
    acc = torch.empty(1, Sq, H, D, device="cuda", dtype=torch.float32)
    lse = torch.empty(1, H, Sq, device="cuda", dtype=torch.float32)
    lcb._lib.attn_fwd_ex(q, k1, v1, acc, lse, False, scale)
    acc2, lse2 = acc.clone(), lse.clone()
    lcb._lib.attn_fwd_ex(q, k2, v2, acc, lse, False, scale, merge=True)
    ob = torch.empty(1, Sq, H, D, device="cuda", dtype=torch.bfloat16)
    lb = torch.empty(1, H, Sq, device="cuda", dtype=torch.float32)
    lcb._lib.attn_fwd_ex(q, k2, v2, ob, lb, False, scale)
    lcb._lib.attn_lse_merge(acc2, lse2, ob, lb)
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.attn_fwd(to64(q), to64(k), to64(v), False, scale)
    assert_bf16_close(to64(acc), ref_o, "O merge mode vs oracle")
    assert_lse_close(to64(lse), ref_lse)
    # the fused form keeps the block in fp32; the unfused one rounds it to bf16 first
    assert_bf16_close(to64(acc), to64(acc2), "O merge mode vs unfused", max_abs=1e-2, mean_abs=1e-3)
    assert_lse_close(to64(lse), to64(lse2), tol=1e-5)


def test_forward_merge_mode_empty_sides():
    """An accumulator row with LSE = -inf (no keys yet) takes the block's result
    whatever its O holds; a block with no keys leaves the accumulator as it was."""
    Sq, Sk, H = 160, 96, 2
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(1, n, H, D, generator=g).to("cuda", torch.bfloat16) for n in (Sq, Sk, Sk))
    scale = D ** -0.5
    acc = torch.full((1, Sq, H, D), float("nan"), device="cuda")
    lse = torch.full((1, H, Sq), float("-inf"), device="cuda")
    lcb._lib.attn_fwd_ex(q, k, v, acc, lse, False, scale, merge=True)
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.attn_fwd(to64(q), to64(k), to64(v), False, scale)
    assert torch.isfinite(acc).all()
    assert_bf16_close(to64(acc), ref_o, "O merge into empty accumulator")
    assert_lse_close(to64(lse), ref_lse)
    before_o, before_l = acc.clone(), lse.clone()
    lcb._lib.attn_fwd_ex(q, k[:, :0], v[:, :0], acc, lse, False, scale, merge=True)
    torch.cuda.synchronize()
    assert torch.equal(acc, before_o) and torch.equal(lse, before_l)


def test_ring_backward_fused_and_two_pass_agree():
    """The ring backward as one-pass tasks (dQ into one tiled accumulator) and
    as deterministic two-pass tasks give the same gradients within bf16
    rounding; dK and dV are bit-identical (same per-task products)."""
    S, H, P = 4096, 2, 4
    q, k, v, do = gaussian_qkvdo(1, H, S, D, seed=78)
    plan = ZigzagPlan(S, P, "cuda")
    qz, kz, vz, doz = (plan.gather(x) for x in (q, k, v, do))
    oz, lsez, _ = lcb.zigzag_attention_fwd(qz, kz, vz, plan)
    g1 = lcb.zigzag_attention_bwd(qz, kz, vz, oz, lsez, doz, plan, fused=True)
    g2 = lcb.zigzag_attention_bwd(qz, kz, vz, oz, lsez, doz, plan, fused=False)
    torch.cuda.synchronize()
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert (g1[0].float() - g2[0].float()).abs().max().item() <= 2 ** -7 * g2[0].float().abs().max().item()
