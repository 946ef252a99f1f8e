"""fp64 oracle for the cross-entropy loss head with an in-place backward.

TEST INFRASTRUCTURE (see the package header): only tests/, the smoke check and
the bench's CPU-baseline leg may call this module.

What the pages fix: the long-context training script computes its loss with
Flash Attention's fused cross-entropy kernel, whose backward writes the
gradient over the logits ("EasyContext内存优化秘籍DeepSpeed Zero3卸载策略详解",
§进阶优化与其他技术结合 1: CrossEntropyLoss(inplace_backward=True)). The loss
itself is the textbook one (the reading taken for the pages' silence), per
token row i with label y_i over a vocabulary of V logits x_i:

    LSE_i   = ln sum_j exp(x_ij)
    loss_i  = LSE_i - x_{i, y_i}
    dx_ij   = g_i (exp(x_ij - LSE_i) - [j == y_i])

for an upstream gradient g_i of loss_i. A row whose label equals ignore_index
has loss 0 and gradient 0 (its LSE is still reported). Every step in fp64;
the only stabilisation is subtracting the row maximum before exp.
"""

import numpy as np


def _rows(logits):
    x = np.asarray(logits, dtype=np.float64)
    if x.ndim != 2:
        raise ValueError("logits must be [N, V]")
    return x


def ce_lse(logits):
    """LSE_i = ln sum_j exp(x_ij), [N]."""
    x = _rows(logits)
    m = x.max(axis=1)
    return m + np.log(np.exp(x - m[:, None]).sum(axis=1))


def ce_fwd(logits, labels, ignore_index=-100):
    """Returns (loss [N], lse [N]) in fp64."""
    x = _rows(logits)
    y = np.asarray(labels, dtype=np.int64)
    lse = ce_lse(x)
    keep = y != ignore_index
    picked = np.where(keep, x[np.arange(len(y)), np.where(keep, y, 0)], 0.0)
    loss = np.where(keep, lse - picked, 0.0)
    return loss, lse


def ce_grad(logits, labels, dloss, ignore_index=-100):
    """dL/dx [N, V] for L = sum_i dloss_i * loss_i."""
    x = _rows(logits)
    y = np.asarray(labels, dtype=np.int64)
    g = np.asarray(dloss, dtype=np.float64) * np.ones(len(y))
    lse = ce_lse(x)
    p = np.exp(x - lse[:, None])
    keep = y != ignore_index
    onehot = np.zeros_like(p)
    onehot[np.arange(len(y))[keep], y[keep]] = 1.0
    grad = g[:, None] * (p - onehot)
    grad[~keep] = 0.0
    return grad
