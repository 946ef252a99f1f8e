"""fp64 oracle for merging two partial attention results by log-sum-exp.

TEST INFRASTRUCTURE (see the package header).

Ring attention ("EasyContext核心技术解析：序列并行与Flash Attention的完美结合",
§1 "序列并行技术"; the zigzag ring of "EasyContext代码解析200行核心训练脚本实现
原理", §模型并行策略解析) computes, at each ring step, attention of the local
queries over one block of keys. Two such partial results (O_a, LSE_a) over key
set A and (O_b, LSE_b) over a disjoint key set B combine into attention over
A ∪ B. With Z_x = exp(LSE_x) the softmax denominator over set x:

    LSE = ln(Z_a + Z_b)
    O   = (Z_a O_a + Z_b O_b) / (Z_a + Z_b)

written with the larger LSE factored out so nothing overflows:

    m   = max(LSE_a, LSE_b),  w_x = exp(LSE_x - m)
    LSE = m + ln(w_a + w_b),  O = (w_a O_a + w_b O_b) / (w_a + w_b)

A side with LSE = -inf has no visible key and weight 0; if both are -inf the
merged row is LSE = -inf, O = 0.
"""

import numpy as np


def lse_merge(o_a, lse_a, o_b, lse_b):
    """Merge row-wise. o_*: [..., R, H, D]; lse_*: [..., H, R] (attention layouts).

    Returns (o, lse) in fp64 with the same shapes.
    """
    o_a, o_b = np.asarray(o_a, np.float64), np.asarray(o_b, np.float64)
    la, lb = np.asarray(lse_a, np.float64), np.asarray(lse_b, np.float64)
    m = np.maximum(la, lb)
    empty = ~np.isfinite(m)
    m0 = np.where(empty, 0.0, m)
    wa = np.where(np.isfinite(la), np.exp(la - m0), 0.0)
    wb = np.where(np.isfinite(lb), np.exp(lb - m0), 0.0)
    den = wa + wb
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(empty, -np.inf, m0 + np.log(np.where(empty, 1.0, den)))
        ca = np.where(empty, 0.0, wa / np.where(empty, 1.0, den))
        cb = np.where(empty, 0.0, wb / np.where(empty, 1.0, den))
    # lse is [..., H, R]; o is [..., R, H, D]: move H behind R for the weights.
    ca_o = np.swapaxes(ca, -1, -2)[..., None]
    cb_o = np.swapaxes(cb, -1, -2)[..., None]
    o = ca_o * o_a + cb_o * o_b
    return o, lse
