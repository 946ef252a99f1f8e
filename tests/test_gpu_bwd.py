"""GPU parity of the backward passes (dK/dV and dQ) against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import long_context_causal_blockwise_gb300 as lcb
from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo, sample_rows
from parity import assert_bf16_close, assert_lse_close, head64, map_heads, rows_budget, to64

pytestmark = pytest.mark.gpu
D = 128


def _bwd_full_check(B, H, S, causal, seed):
    q, k, v, do = gaussian_qkvdo(B, H, S, D, seed=seed)
    o, lse = lcb.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = lcb.attn_bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    ref = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, D ** -0.5)
    tag = f"B{B} H{H} S{S} causal{causal}"
    assert_bf16_close(to64(dq), ref["dq"], "dQ " + tag)
    assert_bf16_close(to64(dk), ref["dk"], "dK " + tag)
    assert_bf16_close(to64(dv), ref["dv"], "dV " + tag)


def test_config1_shape_backward_full_tensors():
    _bwd_full_check(1, 4, 1024, True, seed=0)


@pytest.mark.parametrize("S", [1, 7, 128, 129, 256, 383, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_lengths(S, causal):
    _bwd_full_check(2, 2, S, causal, seed=100 + S)


def test_block_backward_accumulates_to_monolithic():
    """Key blocks with the full problem's LSE/Delta, fp32 accumulate, add up exactly."""
    B, H, Sq, Sk = 1, 2, 256, 640
    g = torch.Generator(device="cuda").manual_seed(3)
    mk = lambda n: torch.randn(B, n, H, D, generator=g, device="cuda").to(torch.bfloat16)  # noqa: E731
    q, k, v, do = mk(Sq), mk(Sk), mk(Sk), mk(Sq)
    o = torch.empty(B, Sq, H, D, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(B, H, Sq, device="cuda")
    lcb.attn_fwd_ex(q, k, v, o, lse, False, D ** -0.5)
    delta = torch.empty(B, H, Sq, device="cuda")
    lcb.attn_bwd_preprocess(o, do, delta)
    dq = torch.zeros(B, Sq, H, D, device="cuda")
    dk = torch.zeros(B, Sk, H, D, device="cuda")
    dv = torch.zeros(B, Sk, H, D, device="cuda")
    cuts = [(0, 200), (200, 456), (456, 640)]
    for a, b in cuts:
        # fp32 accumulate: dq sums over the blocks, each block adds to its own dk/dv rows
        lcb.attn_bwd_ex(q, k[:, a:b], v[:, a:b], lse, delta, do, dq, dk[:, a:b], dv[:, a:b], False, D ** -0.5,
                        accumulate=True)
    torch.cuda.synchronize()
    ref = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), False, D ** -0.5)
    assert_bf16_close(to64(dq), ref["dq"], "dQ blocks")
    assert_bf16_close(to64(dk), ref["dk"], "dK blocks")
    assert_bf16_close(to64(dv), ref["dv"], "dV blocks")
    # fp32 store mode overwrites: a second pass over one block in store mode equals that block alone
    dk2 = torch.full_like(dk[:, :200], 9.0)
    dv2 = torch.full_like(dv[:, :200], 9.0)
    dq2 = torch.full_like(dq, 9.0)
    lcb.attn_bwd_ex(q, k[:, :200], v[:, :200], lse, delta, do, dq2, dk2, dv2, False, D ** -0.5, accumulate=False)
    torch.cuda.synchronize()
    assert torch.equal(dk2, dk[:, :200]) and torch.equal(dv2, dv[:, :200])


def test_split_passes_match_combined():
    B, H, S = 1, 2, 512
    q, k, v, do = gaussian_qkvdo(B, H, S, D, seed=8)
    o, lse = lcb.attn_fwd(q, k, v)
    delta = torch.empty(B, H, S, device="cuda")
    lcb.attn_bwd_preprocess(o, do, delta)
    g1 = [torch.empty_like(q) for _ in range(3)]
    g2 = [torch.full_like(q, 3.0) for _ in range(3)]
    lcb.attn_bwd_ex(q, k, v, lse, delta, do, *g1, True, D ** -0.5)
    lcb.attn_bwd_ex(q, k, v, lse, delta, do, *g2, True, D ** -0.5, passes="dkdv")
    torch.cuda.synchronize()
    assert torch.equal(g2[1], g1[1]) and torch.equal(g2[2], g1[2])
    assert (g2[0] == 3.0).all()  # dq untouched by the dK/dV pass
    lcb.attn_bwd_ex(q, k, v, lse, delta, do, *g2, True, D ** -0.5, passes="dq")
    torch.cuda.synchronize()
    assert torch.equal(g2[0], g1[0])


def test_empty_sides():
    """Sk = 0: dQ is zero; Sq = 0: dK and dV are zero."""
    B, H = 1, 2
    q = torch.randn(B, 64, H, D, device="cuda").to(torch.bfloat16)
    e = torch.empty(B, 0, H, D, device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros(B, H, 64, device="cuda")
    delta = torch.zeros(B, H, 64, device="cuda")
    dq = torch.full_like(q, 5.0)
    lcb.attn_bwd_ex(q, e, e, lse, delta, q, dq, e, e, False, D ** -0.5)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dq) == 0
    dk = torch.full_like(q, 5.0)
    dv = torch.full_like(q, 5.0)
    le = torch.zeros(B, H, 0, device="cuda")
    lcb.attn_bwd_ex(e, q, q, le, le, e, e, dk, dv, False, D ** -0.5)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0


def test_config2_sampled_rows_backward():
    """B=1, H=32, S=32768: O, LSE and dQ on 4096 sampled query rows of every
    head; dK/dV on 4096 sampled key rows of two heads; the sum invariants on
    every head."""
    B, H, S = 1, 32, 32768
    scale = D ** -0.5
    q, k, v, do = gaussian_qkvdo(B, H, S, D, seed=0)
    o, lse = lcb.attn_fwd(q, k, v)
    dq, dk, dv = lcb.attn_bwd(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    rows = sample_rows(S, rows_budget(4096), seed=1)
    refs = map_heads(lambda h: oracle.attn_rows(*(head64(t, h) for t in (q, k, v, do)), rows, True, scale),
                     list(range(H)))
    rows_d = torch.as_tensor(rows, device="cuda")
    assert_bf16_close(to64(o[:, rows_d]), np.concatenate([r["o"] for r in refs], 2), "O C2 sampled")
    assert_lse_close(to64(lse[:, :, rows_d]), np.concatenate([r["lse"] for r in refs], 1))
    assert_bf16_close(to64(dq[:, rows_d]), np.concatenate([r["dq"] for r in refs], 2), "dQ C2 sampled")
    keys = sample_rows(S, rows_budget(4096), seed=2)
    keys_d = torch.as_tensor(keys, device="cuda")
    heads = [0, 31]
    kref = map_heads(lambda h: oracle.attn_key_rows(*(head64(t, h) for t in (q, k, v, do)), keys, [0], True, scale),
                     heads)
    for h, (rdk, rdv) in zip(heads, kref):
        assert_bf16_close(to64(dk[:, keys_d, h:h + 1]), rdk, f"dK C2 sampled head {h}")
        assert_bf16_close(to64(dv[:, keys_d, h:h + 1]), rdv, f"dV C2 sampled head {h}")
    # sum_j dV_j = sum_i dO_i and sum_j dK_j = 0, per head (fp32 sums of bf16 values)
    sdv = dv.float().sum(1)
    sdo = do.float().sum(1)
    sdk = dk.float().sum(1)
    tol = 1e-2 * sdo.norm(dim=-1, keepdim=True)
    assert ((sdv - sdo).norm(dim=-1, keepdim=True) <= tol).all()
    assert (sdk.norm(dim=-1) <= 1e-2 * dk.float().norm(dim=(1, 3))).all()
