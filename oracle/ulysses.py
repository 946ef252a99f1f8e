"""Oracle for Ulysses sequence parallelism: the sequence <-> head all-to-all.

TEST INFRASTRUCTURE (see the package header).

The pages name Ulysses attention as one of the sequence-parallel modes
("EasyContext核心技术解析：序列并行与Flash Attention的完美结合", §1 "序列并行技术":
Ulysses注意力, based on DeepSpeed; "EasyContext代码解析200行核心训练脚本实现原理",
§模型并行策略解析: ulysses_attn; "EasyContext未来展望：从1M到10M上下文的技术路线图",
§关键技术突破点: Deepspeed Ulysses) without spelling out its steps. The plain
reading, the DeepSpeed-Ulysses method, is taken here:

  * P ranks; the sequence of S tokens is cut into P contiguous pieces of
    S / P tokens, rank r holding rows [r S/P, (r+1) S/P) of every head;
  * an all-to-all over the heads: the H heads are cut into P groups of
    H / P, and rank r sends group j of its rows to rank j, which places them
    at rows [r S/P, (r+1) S/P). Afterwards rank j holds ALL S rows of head
    group j;
  * each rank computes ordinary (causal) attention for its H / P heads over
    the whole sequence;
  * the inverse all-to-all returns the output to the sequence pieces.

Attention is independent per head, so the result equals attention over all
heads at once: the all-to-all moves data and does no arithmetic.
"""

import numpy as np

from .attention import attn_fwd


def _check(S, H, P):
    if P < 1 or H % P != 0 or S % P != 0:
        raise ValueError("Ulysses needs P >= 1 dividing both H and S")


def seq_to_head(x, P):
    """All-to-all, sequence pieces -> head groups.

    x: [B, S, H, D], the concatenation of the P ranks' pieces (rank r's rows
    [r S/P, (r+1) S/P)). Returns a list of P arrays, rank j's [B, S, H/P, D]
    (all rows of head group j)."""
    B, S, H, D = x.shape
    _check(S, H, P)
    n, hp = S // P, H // P
    out = [np.empty((B, S, hp, D), dtype=x.dtype) for _ in range(P)]
    for r in range(P):          # sender: rank r's sequence piece
        piece = x[:, r * n:(r + 1) * n]
        for j in range(P):      # receiver: rank j takes head group j of it
            out[j][:, r * n:(r + 1) * n] = piece[:, :, j * hp:(j + 1) * hp]
    return out


def head_to_seq(parts, P):
    """The inverse all-to-all: P arrays [B, S, H/P, D] -> [B, S, H, D]."""
    if len(parts) != P:
        raise ValueError("one array per rank")
    B, S, hp, D = parts[0].shape
    H = hp * P
    _check(S, H, P)
    n = S // P
    x = np.empty((B, S, H, D), dtype=parts[0].dtype)
    for j in range(P):          # sender: rank j's head group, every row
        for r in range(P):      # receiver: rank r takes its own rows of it
            x[:, r * n:(r + 1) * n, j * hp:(j + 1) * hp] = parts[j][:, r * n:(r + 1) * n]
    return x


def ulysses_attn_fwd(q, k, v, P, causal, scale):
    """Ulysses attention on P ranks: all-to-all of Q, K, V, attention of each
    rank's head group over the whole sequence, inverse all-to-all of O.
    Returns (O [B, S, H, D], LSE [B, H, S]) in the monolithic layout."""
    qs, ks, vs = seq_to_head(q, P), seq_to_head(k, P), seq_to_head(v, P)
    outs, lses = [], []
    for j in range(P):
        o_j, lse_j = attn_fwd(qs[j], ks[j], vs[j], causal, scale)
        outs.append(o_j)
        lses.append(lse_j)
    return head_to_seq(outs, P), np.concatenate(lses, axis=1)
