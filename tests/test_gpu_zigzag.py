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
from parity import assert_bf16_close, assert_lse_close, to64

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
    on every element, and vs the oracle on sampled query rows."""
    S, H, P = 131072, 32, 8
    r = _run(S, H, P, seed=0)
    _vs_monolithic(r, "C3")
    rows = sample_rows(S, 48, seed=3)
    # chunk edges of the zigzag split are among the most likely places to go wrong
    c = S // (2 * P)
    rows = np.unique(np.concatenate([rows, [c - 1, c, 7 * c - 1, 7 * c, 8 * c, 15 * c - 1]]))
    ref = oracle.attn_rows(to64(r["q"]), to64(r["k"]), to64(r["v"]), to64(r["do"]), rows, True, D ** -0.5)
    inv = np.argsort(np.asarray(r["plan"].perm))
    zpos = torch.as_tensor(inv[rows], device="cuda")
    assert_bf16_close(to64(r["oz"][:, zpos]), ref["o"], "O C3 sampled vs oracle")
    assert_lse_close(to64(r["lsez"][:, :, zpos]), ref["lse"])
    assert_bf16_close(to64(r["dqz"][:, zpos]), ref["dq"], "dQ C3 sampled vs oracle")
