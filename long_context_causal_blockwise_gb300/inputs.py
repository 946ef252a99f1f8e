"""Seeded synthetic inputs shaped like Llama-2 attention layers.

This module holds no attention arithmetic. It only draws the random inputs
that both the CUDA path and the oracle read, so both see identical bf16
values (the oracle gets a host copy, upcast to fp64):

  * Q, K, V, dO: i.i.d. N(0, 1), drawn in fp32 from one torch.Generator seeded
    with `seed`, in the order Q, K, V, dO, then rounded to bf16.
  * Optional RoPE pre-rotation of Q and K (the long-context recipe raises the
    rotary base, "EasyContext核心技术解析：序列并行与Flash Attention的完美结合"
    §3 "RoPE扩展技术" and the --rope-theta 1000000 flag of the training script
    on "EasyContext内存优化秘籍DeepSpeed Zero3卸载策略详解"): rotate-half
    pairing (d, d + D/2), inv_freq_k = theta^(-2k/D), angles pos * inv_freq in
    fp64, applied to the fp32 draws and rounded to bf16 once. Rotating
    i.i.d. Gaussian pairs leaves them i.i.d. N(0, 1).
  * sample_rows: deterministic sampled query rows for large problems (first
    and last row, tile edges 128k-1 / 128k, the rest uniform from the seed).
"""

import numpy as np
import torch


def gaussian_qkvdo(B, H, S, D, seed=0, device="cuda", rope_theta=None, with_do=True):
    """Returns (q, k, v, do) bf16 [B, S, H, D] tensors on `device` (do may be None)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    shape = (B, S, H, D)
    out = []
    names = ("q", "k", "v", "do") if with_do else ("q", "k", "v")
    for name in names:
        x = torch.randn(shape, generator=gen, dtype=torch.float32, device=dev)
        if rope_theta is not None and name in ("q", "k"):
            x = _rope_fp32(x, float(rope_theta))
        out.append(x.to(torch.bfloat16))
        del x
    if not with_do:
        out.append(None)
    return tuple(out)


def _rope_fp32(x, theta, chunk=1 << 16):
    """Rotate-half RoPE along D with positions 0..S-1; angles in fp64."""
    B, S, H, D = x.shape
    half = D // 2
    inv_freq = theta ** (-torch.arange(0, half, dtype=torch.float64, device=x.device) * 2.0 / D)
    y = torch.empty_like(x)
    for s0 in range(0, S, chunk):
        s1 = min(S, s0 + chunk)
        pos = torch.arange(s0, s1, dtype=torch.float64, device=x.device)
        ang = pos[:, None] * inv_freq[None, :]
        cos = torch.cos(ang)[None, :, None, :]
        sin = torch.sin(ang)[None, :, None, :]
        a = x[:, s0:s1, :, :half].to(torch.float64)
        b = x[:, s0:s1, :, half:].to(torch.float64)
        y[:, s0:s1, :, :half] = (a * cos - b * sin).to(torch.float32)
        y[:, s0:s1, :, half:] = (b * cos + a * sin).to(torch.float32)
    return y


def sample_rows(S, n, seed=0, tile=128):
    """Sorted unique row indices: 0, S-1, tile edges, then uniform draws."""
    rng = np.random.default_rng(int(seed) + 7919)
    rows = {0, S - 1}
    edge_budget = n // 4
    k = 1
    while len(rows) < edge_budget and k * tile < S:
        rows.add(k * tile - 1)
        rows.add(k * tile)
        k += max(1, (S // tile) // max(1, edge_budget // 2))
    n = min(n, S)
    while len(rows) < n:
        rows.update(int(r) for r in rng.integers(0, S, size=n - len(rows)))
    return np.array(sorted(rows)[:n] if len(rows) > n else sorted(rows), dtype=np.int64)
