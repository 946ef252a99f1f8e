"""fp64 oracle for rotary position embedding (RoPE) with a raised base.

TEST INFRASTRUCTURE (see the package header): only tests/, the smoke check and
the bench's CPU-baseline leg may call this module.

What the pages fix: long-context training raises the model's rotary base
theta ("EasyContext核心技术解析：序列并行与Flash Attention的完美结合",
§3 "RoPE扩展技术"; the --rope-theta 1000000 flag on "EasyContext内存优化秘籍
DeepSpeed Zero3卸载策略详解", §训练脚本配置; the base raised step-wise to 1e9
on "EasyContext：用最少资源扩展大模型至百万Token"). The rotation itself is the
one of the Llama attention those pages train (the reading taken for the
pages' silence): for head dimension D, pair k = 0 .. D/2 - 1 couples features
k and k + D/2 and turns by angle a = (pos0 + i) * theta^(-2k/D) at token i:

    y_k         = x_k cos a - x_{k+D/2} sin a
    y_{k+D/2}   = x_{k+D/2} cos a + x_k sin a

A rotation's inverse is its transpose, the turn by -a; it maps a gradient
with respect to the rotated tensor back to the unrotated one.
Layout [B, S, H, D]; every step in fp64.
"""

import numpy as np


def rope(x, theta, pos0=0, inverse=False):
    """Rotate x [B, S, H, D] (any float dtype; computed in fp64) by RoPE."""
    x = np.asarray(x, dtype=np.float64)
    if x.ndim != 4 or x.shape[3] % 2:
        raise ValueError("x must be [B, S, H, D] with D even")
    S, D = x.shape[1], x.shape[3]
    half = D // 2
    freq = float(theta) ** (-2.0 * np.arange(half, dtype=np.float64) / D)
    pos = float(pos0) + np.arange(S, dtype=np.float64)
    ang = pos[:, None] * freq[None, :]  # [S, D/2]
    if inverse:
        ang = -ang
    c = np.cos(ang)[None, :, None, :]
    s = np.sin(ang)[None, :, None, :]
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)
