"""GPU parity of the RoPE kernel (raised rotary base) against the fp64 oracle,
alone and as the rotation around causal attention (forward and backward)."""

import numpy as np
import pytest
import torch

import oracle
import long_context_causal_blockwise_gb300 as lcb
from parity import assert_bf16_close, assert_lse_close, to64

pytestmark = pytest.mark.gpu
D = 128


def _rope_err(got, want, x):
    """|got - want| over its bound: one bf16 step at |want| (the output rounding
    and a boundary case) plus 1e-6 (|x_k| + |x_k+64|) for the fp32 sin/cos and
    rotation (about 3e-7 of the pair's size)."""
    a = np.abs(want)
    step = 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -120))) - 7)
    pair = np.abs(x[..., :64]) + np.abs(x[..., 64:])
    bound = step + 1e-6 * np.concatenate([pair, pair], axis=-1)
    return np.abs(got - want) / bound


@pytest.mark.parametrize("theta,pos0", [(1e4, 0), (1e6, 0), (1e6, 500_000), (1e9, 1_000_000), (1e6, 1_000_000_000)])
def test_rope_matches_oracle(theta, pos0):
    """Every element within one bf16 step of the fp64 rotation rounded to bf16,
    almost all of them equal; the inverse undoes it within bf16 rounding."""
    g = torch.Generator(device="cuda").manual_seed(int(theta) % 1000 + pos0 % 997)
    x = torch.randn(2, 777, 3, D, generator=g, device="cuda").to(torch.bfloat16)
    y = lcb.rope(x, theta, pos0, out=torch.empty_like(x))
    torch.cuda.synchronize()
    want = oracle.rope(to64(x), theta, pos0)
    err = _rope_err(to64(y), want, to64(x))
    assert err.max() <= 1.0, err.max()
    # almost every element is the exact rotation rounded to bf16
    exact = torch.as_tensor(want).to(torch.bfloat16).double().numpy()
    assert (to64(y) != exact).mean() < 1e-3
    back = lcb.rope(y.clone(), theta, pos0, inverse=True)  # in place on a copy
    torch.cuda.synchronize()
    assert np.abs(to64(back) - to64(x)).max() <= 2.0 ** -6 * np.abs(to64(x)).max()


@pytest.mark.parametrize("H,in_place", [(8, False), (11, True), (32, True), (40, False)])
def test_rope_head_batches_match_oracle(H, in_place):
    """Head counts the kernel takes in batches of eight loads before their
    stores (8, 32, 40) and with a remainder after them (11), in place and not:
    every element within the bound of the fp64 rotation."""
    g = torch.Generator(device="cuda").manual_seed(H)
    x = torch.randn(1, 129, H, D, generator=g, device="cuda").to(torch.bfloat16)
    want = oracle.rope(to64(x), 1e6, 4096)
    x_before = to64(x)
    y = lcb.rope(x, 1e6, 4096) if in_place else lcb.rope(x, 1e6, 4096, out=torch.empty_like(x))
    torch.cuda.synchronize()
    assert _rope_err(to64(y), want, x_before).max() <= 1.0
    if in_place:
        assert y.data_ptr() == x.data_ptr()


def test_rope_strided_view_and_in_place():
    """Row strides wider than H*D (a q slice of a packed qkv buffer) and x == out."""
    g = torch.Generator(device="cuda").manual_seed(5)
    qkv = torch.randn(1, 300, 3, 2, D, generator=g, device="cuda").to(torch.bfloat16)
    q = qkv[:, :, 0]  # [1, 300, 2, 128], row stride 3*2*128
    q_before = to64(q)
    ref = oracle.rope(q_before, 1e6, 1234)
    k_before = qkv[:, :, 1].clone()
    lcb.rope(q, 1e6, 1234)
    torch.cuda.synchronize()
    assert _rope_err(to64(qkv[:, :, 0]), ref, q_before).max() <= 1.0
    assert torch.equal(qkv[:, :, 1], k_before)


def test_rope_attention_forward_backward_vs_oracle():
    """Raw q, k -> RoPE -> causal attention -> RoPE^T on dQ, dK, at the end of a
    512K context (positions 523264 .. 524287, theta = 1e6), against the fp64
    oracle of the same chain (the rotated q, k rounded to bf16, as the kernel's
    output is)."""
    B, H, S = 1, 2, 1024
    pos0 = 524288 - S
    theta = 1e6
    scale = D ** -0.5
    g = torch.Generator(device="cuda").manual_seed(12)
    q, k, v, do = (torch.randn(B, S, H, D, generator=g, device="cuda").to(torch.bfloat16) for _ in range(4))
    qr = lcb.rope(q, theta, pos0, out=torch.empty_like(q))
    kr = lcb.rope(k, theta, pos0, out=torch.empty_like(k))
    o, lse = lcb.attn_fwd(qr, kr, v)
    dqr, dkr, dv = lcb.attn_bwd(qr, kr, v, o, lse, do)
    dq = lcb.rope(dqr, theta, pos0, inverse=True, out=torch.empty_like(dqr))
    dk = lcb.rope(dkr, theta, pos0, inverse=True, out=torch.empty_like(dkr))
    torch.cuda.synchronize()
    # lcb_rope's output is the rotation rounded to bf16 once; attention reads those values
    q64, k64 = (to64(torch.as_tensor(oracle.rope(to64(t), theta, pos0)).to(torch.bfloat16)) for t in (q, k))
    ref = oracle.attn_bwd(q64, k64, to64(v), to64(do), True, scale)
    assert_bf16_close(to64(o), ref["o"], "O (RoPE)")
    assert_lse_close(to64(lse), ref["lse"])
    assert_bf16_close(to64(dq), oracle.rope(ref["dq"], theta, pos0, inverse=True), "dQ (RoPE^T)")
    assert_bf16_close(to64(dk), oracle.rope(ref["dk"], theta, pos0, inverse=True), "dK (RoPE^T)")
    assert_bf16_close(to64(dv), ref["dv"], "dV (RoPE)")
