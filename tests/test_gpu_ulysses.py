"""Ulysses sequence parallelism emulated on one GPU.

The all-to-all kernel must move every element exactly where the oracle's
all-to-all puts it (bit-exact: it is a copy), and Ulysses attention (the
all-to-all around attention on the head layout) must reproduce monolithic
attention on the GPU and the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import long_context_causal_blockwise_gb300 as lcb
from long_context_causal_blockwise_gb300 import _lib
from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo, sample_rows
from long_context_causal_blockwise_gb300.ulysses import lse_to_monolithic
from parity import assert_bf16_close, assert_lse_close, oracle_rows_by_head, rows_budget, to64

pytestmark = pytest.mark.gpu
D = 128


@pytest.mark.parametrize("B,S,H,P,dtype", [
    (1, 8, 4, 2, torch.bfloat16), (1, 4096, 32, 8, torch.bfloat16), (2, 1000, 40, 8, torch.bfloat16),
    (3, 96, 6, 3, torch.float32), (1, 128, 8, 1, torch.bfloat16), (1, 64, 16, 16, torch.bfloat16),
    (2, 96, 12, 4, torch.float32)])
def test_all_to_all_bit_exact_vs_oracle(B, S, H, P, dtype):
    g = torch.Generator(device="cuda").manual_seed(S * H + P)
    x = torch.randn(B, S, H, D, generator=g, device="cuda").to(dtype)
    xh = lcb.ulysses_all_to_all(x, P, to_heads=True)
    back = lcb.ulysses_all_to_all(xh, P, to_heads=False)
    torch.cuda.synchronize()
    want = oracle.ulysses_seq_to_head(x.cpu().numpy() if dtype == torch.float32 else
                                      x.view(torch.int16).cpu().numpy(), P)
    got = xh.cpu().numpy() if dtype == torch.float32 else xh.view(torch.int16).cpu().numpy()
    for j in range(P):  # rank j's part: rows [j B, (j+1) B) of the head-layout batch
        assert np.array_equal(got[j * B:(j + 1) * B], want[j]), f"rank {j}"
    assert torch.equal(back, x)


def test_all_to_all_argument_errors():
    lib = _lib.load()
    x = torch.zeros(1, 16, 8, D, device="cuda", dtype=torch.bfloat16)
    y = torch.empty_like(x)
    p = lambda t: t.data_ptr()  # noqa: E731
    assert lib.lcb_ulysses_all_to_all(p(x), p(y), 1, 16, 8, D, 3, 2, 0, None) == _lib.LCB_ERR_ARG  # 3 does not divide 8
    assert lib.lcb_ulysses_all_to_all(p(x), p(y), 1, 16, 8, D, 2, 3, 0, None) == _lib.LCB_ERR_UNSUPPORTED
    assert lib.lcb_ulysses_all_to_all(p(x), p(x), 1, 16, 8, D, 2, 2, 0, None) == _lib.LCB_ERR_ARG  # in place
    assert lib.lcb_ulysses_all_to_all(p(x), p(y), 1, 16, 8, D, 2, 2, 2, None) == _lib.LCB_ERR_ARG  # direction
    assert lib.lcb_ulysses_all_to_all(p(x), p(y), 1, 16, 8, 4, 8, 2, 0, None) == _lib.LCB_ERR_ARG  # 8-byte blocks


def _ulysses_vs_monolithic(B, S, H, P, causal, seed):
    q, k, v, do = gaussian_qkvdo(B, H, S, D, seed=seed)
    o_u, ctx = lcb.ulysses_attention_fwd(q, k, v, P, causal=causal)
    dq_u, dk_u, dv_u = lcb.ulysses_attention_bwd(do, ctx)
    o, lse = lcb.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = lcb.attn_bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    # every head is computed by the same kernel code on the same values: O, LSE,
    # dK, dV bit for bit; dQ (fp32 sums in no fixed order) within bf16 rounding
    assert torch.equal(o_u, o)
    assert torch.equal(lse_to_monolithic(ctx.lse, P), lse)
    assert torch.equal(dk_u, dk) and torch.equal(dv_u, dv)
    assert (dq_u.float() - dq.float()).abs().max().item() <= 2 ** -7 * dq.float().abs().max().item()
    return q, k, v, do, o_u, ctx, dq_u, dk_u, dv_u


@pytest.mark.parametrize("B,S,H,P,causal", [(1, 1024, 8, 4, True), (2, 768, 6, 3, False), (1, 640, 4, 1, True)])
def test_ulysses_attention_vs_monolithic_and_oracle(B, S, H, P, causal):
    q, k, v, do, o_u, ctx, dq_u, dk_u, dv_u = _ulysses_vs_monolithic(B, S, H, P, causal, seed=S + P)
    ref = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, D ** -0.5)
    o_ref, lse_ref = oracle.ulysses_attn_fwd(to64(q), to64(k), to64(v), P, causal, D ** -0.5)
    assert_bf16_close(to64(o_u), o_ref, "O Ulysses vs oracle")
    assert_lse_close(to64(lse_to_monolithic(ctx.lse, P)), lse_ref)
    assert_bf16_close(to64(dq_u), ref["dq"], "dQ Ulysses vs oracle")
    assert_bf16_close(to64(dk_u), ref["dk"], "dK Ulysses vs oracle")
    assert_bf16_close(to64(dv_u), ref["dv"], "dV Ulysses vs oracle")


def test_ulysses_131072_p8():
    """B=1, H=32, S=131072 over P=8 ranks (4 heads each): the result equals
    monolithic attention (bit for bit but dQ), and O, LSE, dQ agree with the
    oracle on sampled query rows of every head."""
    S, H, P = 131072, 32, 8
    q, k, v, do, o_u, ctx, dq_u, _, _ = _ulysses_vs_monolithic(1, S, H, P, True, seed=0)
    rows = sample_rows(S, rows_budget(1024), seed=11)
    # the sequence pieces' edges, where a misplaced row would show first
    n = S // P
    rows = np.unique(np.concatenate([rows, [e for r in range(1, P) for e in (r * n - 1, r * n)]]))
    refs = oracle_rows_by_head(q, k, v, do, rows, True, D ** -0.5)
    idx = torch.as_tensor(rows, device="cuda")
    assert_bf16_close(to64(o_u[:, idx]), np.concatenate([x["o"] for x in refs], 2), "O Ulysses sampled vs oracle")
    assert_lse_close(to64(lse_to_monolithic(ctx.lse, P)[:, :, idx]), np.concatenate([x["lse"] for x in refs], 1))
    assert_bf16_close(to64(dq_u[:, idx]), np.concatenate([x["dq"] for x in refs], 2), "dQ Ulysses sampled vs oracle")
