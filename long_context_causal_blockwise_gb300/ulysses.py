"""Ulysses sequence parallelism emulated on one GPU.

Ulysses attention ("EasyContext核心技术解析：序列并行与Flash Attention的完美结合",
§1 "序列并行技术": Ulysses注意力, based on DeepSpeed;
"EasyContext代码解析200行核心训练脚本实现原理", §模型并行策略解析: ulysses_attn)
keeps each of P ranks' sequence piece of all heads, and around attention
swaps the sharding with an all-to-all: afterwards rank j holds the whole
sequence of heads [j H/P, (j+1) H/P) and computes ordinary attention for them.

Here the P ranks are virtual, on one device. The all-to-all is the library's
lcb_ulysses_all_to_all kernel; its head layout is one [P*B, S, H/P, D] tensor,
so every rank's attention runs in a single attn_fwd / attn_bwd call with
batch P*B. Every step runs in libattn.so kernels:

  forward   all-to-all of Q, K, V to the head layout; attn_fwd (batch P*B,
            H/P heads); all-to-all of O back to the sequence layout
  backward  all-to-all of dO to the head layout; attn_bwd on the head layout
            (Q, K, V, O, LSE of the forward kept there, as each rank would
            keep its own); all-to-all of dQ, dK, dV back

LSE stays in the head layout, [P*B, H/P, S]: rank j's statistics for its
heads, which is all its backward needs.
"""

from dataclasses import dataclass

import torch

from . import _lib


@dataclass
class UlyssesCtx:
    """What each rank keeps from the forward for its backward (head layout)."""
    P: int
    causal: bool
    scale: float
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    o: torch.Tensor
    lse: torch.Tensor


def ulysses_attention_fwd(q, k, v, P, causal=True, scale=None, out=None):
    """Attention of [B, S, H, D] bf16 inputs over P emulated Ulysses ranks.

    Returns (o [B, S, H, D] in the sequence layout, ctx) where ctx holds the
    head-layout tensors and LSE [P*B, H/P, S] for the backward."""
    B, S, H, D = q.shape
    scale = D ** -0.5 if scale is None else scale
    qh, kh, vh = (_lib.ulysses_all_to_all(x, P, to_heads=True) for x in (q, k, v))
    oh, lse = _lib.attn_fwd(qh, kh, vh, causal=causal, scale=scale)
    o = _lib.ulysses_all_to_all(oh, P, to_heads=False, out=out)
    return o, UlyssesCtx(P, causal, scale, qh, kh, vh, oh, lse)


def ulysses_attention_bwd(do, ctx, workspace=None):
    """Gradients (dq, dk, dv) [B, S, H, D] bf16 of the forward that made ctx."""
    P = ctx.P
    doh = _lib.ulysses_all_to_all(do, P, to_heads=True)
    dqh, dkh, dvh = _lib.attn_bwd(ctx.q, ctx.k, ctx.v, ctx.o, ctx.lse, doh, causal=ctx.causal, scale=ctx.scale,
                                  workspace=workspace)
    return tuple(_lib.ulysses_all_to_all(g, P, to_heads=False) for g in (dqh, dkh, dvh))


def lse_to_monolithic(lse_h, P):
    """Head-layout LSE [P*B, H/P, S] viewed as [B, H, S] (a copy; for checks)."""
    PB, Hp, S = lse_h.shape
    return lse_h.view(P, PB // P, Hp, S).permute(1, 0, 2, 3).reshape(PB // P, P * Hp, S)
