"""Zigzag ring attention emulated on one GPU.

Zigzag ring attention ("EasyContext代码解析200行核心训练脚本实现原理",
§模型并行策略解析 zigzag_ring_attn; the per-rank split of §训练循环核心逻辑)
gives each of P ranks two of the 2P sequence chunks, r and 2P-1-r, and moves
keys/values around a ring for P steps. Ring steps compose by merging partial
(O, LSE) results ("EasyContext核心技术解析：序列并行与Flash Attention的完美结合",
§1 "序列并行技术").

Here the P ranks are virtual: every rank's data lives in one device's memory in
zigzag order (rank-major), a ring "transfer" is a pointer to the owner's rows,
and no collective runs. Steps are executed step-major (all ranks' step 0, then
step 1, ...), as the real ring would run them in parallel. Every piece of
arithmetic runs in libattn.so kernels:

  forward  one attn_fwd_group launch per ring step s, its P tasks side by side:
           s = 0 (DIAG): causal, writing the fp32 accumulator;
           s > 0       : merge mode, folding each block into the fp32
                         accumulator in the kernel epilogue
           (unfused: attn_fwd_ex per task, a bf16 block result, then
           attn_lse_merge)
           end          : lcb_cast_f32_bf16 of the accumulator
  backward Delta from the final bf16 O (attn_bwd_preprocess), then per ring
           step one grouped one-pass launch (attn_bwd_fused_group) of its P
           tasks, each with the rank's FINAL
           merged LSE and Delta; dK/dV in fp32, stored at step 0 and
           accumulated after into the owning rank's rows; dQ added into the
           querying rank's tiles of one zeroed tiled accumulator; a cast
           (lcb_dq_untile for dQ) to bf16 ends it.

Outputs stay in zigzag order, the layout each rank would hold.
"""

import torch

from . import _lib


class ZigzagPlan:
    """Schedule of one (S, P) zigzag ring and the gather into zigzag order."""

    def __init__(self, S, P, device):
        perm, tasks = _lib.zigzag_schedule(S, P)
        self.S, self.P = S, P
        self.c = S // (2 * P)
        self.perm = perm
        self.tasks = tasks
        self.perm_dev = torch.tensor(perm, dtype=torch.int32, device=device)
        # step-major order: every rank's step s before any rank's step s + 1
        self.order = sorted(tasks, key=lambda t: (t["step"], t["rank"]))

    def gather(self, x):
        """[1, S, H, D] natural order -> zigzag order (a new tensor)."""
        out = torch.empty_like(x)
        return _lib.permute_rows(x, out, self.perm_dev, scatter=False)

    def scatter(self, x):
        """zigzag order -> natural order (a new tensor)."""
        out = torch.empty_like(x)
        return _lib.permute_rows(x, out, self.perm_dev, scatter=True)


def zigzag_attention_fwd(qz, kz, vz, plan, scale=None, o_acc=None, lse=None, o_blk=None, lse_blk=None, o=None,
                         fused=True):
    """Forward of the emulated ring on zigzag-ordered [1, S, H, D] bf16 inputs.

    Returns (o bf16, lse fp32 [1, H, S], o_acc fp32), all in zigzag order.
    fused=True runs each ring step as ONE grouped launch of its P tasks
    (attn_fwd_group) that merges into the accumulator in the kernel epilogue;
    False runs one launch per task, writing the block result, then the
    separate merge kernel.
    Buffers may be passed in to keep allocation out of a timed loop.
    """
    B, S, H, D = qz.shape
    if B != 1 or S != plan.S:
        raise ValueError("zigzag emulation takes B = 1 and the plan's S")
    scale = D ** -0.5 if scale is None else scale
    dev = qz.device
    c2 = 2 * plan.c
    o_acc = torch.empty((1, S, H, D), dtype=torch.float32, device=dev) if o_acc is None else o_acc
    lse = torch.empty((1, H, S), dtype=torch.float32, device=dev) if lse is None else lse
    o_blk = torch.empty((1, c2, H, D), dtype=torch.bfloat16, device=dev) if o_blk is None else o_blk
    lse_blk = torch.empty((1, H, c2), dtype=torch.float32, device=dev) if lse_blk is None else lse_blk
    o = torch.empty_like(qz) if o is None else o
    if fused:
        # one launch per ring step: the P ranks' tasks of a step own disjoint query rows
        for step in range(plan.P):
            tasks = [(t["q_off"], t["q_len"], t["k_off"], t["k_len"], t["causal"], "f32" if step == 0 else "merge")
                     for t in plan.order if t["step"] == step]
            _lib.attn_fwd_group(qz, kz, vz, o_acc, lse, tasks, scale)
    else:
        for t in plan.order:
            qs = slice(t["q_off"], t["q_off"] + t["q_len"])
            ks = slice(t["k_off"], t["k_off"] + t["k_len"])
            if t["step"] == 0:
                _lib.attn_fwd_ex(qz[:, qs], kz[:, ks], vz[:, ks], o_acc[:, qs], lse[:, :, qs], True, scale)
            else:
                n = t["q_len"]
                _lib.attn_fwd_ex(qz[:, qs], kz[:, ks], vz[:, ks], o_blk[:, :n], lse_blk[:, :, :n], False, scale)
                _lib.attn_lse_merge(o_acc[:, qs], lse[:, :, qs], o_blk[:, :n], lse_blk[:, :, :n])
    _lib.cast_f32_bf16(o_acc, o)
    return o, lse, o_acc


def zigzag_attention_bwd(qz, kz, vz, oz, lse, doz, plan, scale=None, delta=None, grads32=None, grads=None,
                         fused=True, dq_tiles=None):
    """Backward of the emulated ring; all tensors in zigzag order.

    fused=True runs each ring step as ONE grouped one-pass launch
    (attn_bwd_group), every task adding its dQ into one tiled fp32
    accumulator (needs chunks of a multiple of 128 rows); otherwise, or with
    fused=False, each task runs as the deterministic two-pass form.
    Returns (dq, dk, dv) bf16 [1, S, H, D].
    """
    B, S, H, D = qz.shape
    scale = D ** -0.5 if scale is None else scale
    dev = qz.device
    fused = fused and plan.c % 128 == 0  # query blocks must start on accumulator tiles
    delta = torch.empty((1, H, S), dtype=torch.float32, device=dev) if delta is None else delta
    if grads32 is None:
        grads32 = tuple(torch.empty((1, S, H, D), dtype=torch.float32, device=dev) for _ in range(3))
    if grads is None:
        grads = tuple(torch.empty_like(qz) for _ in range(3))
    dq32, dk32, dv32 = grads32
    _lib.attn_bwd_preprocess(oz, doz, delta)
    if fused:
        if dq_tiles is None:
            dq_tiles = _lib.dq_tiles_zeros(1, H, S, dev)
        else:
            _lib.dq_tiles_zero_(dq_tiles)  # the fused pass only ever adds into dQ
    if fused:
        # one launch per ring step: the P ranks' tasks of a step own disjoint key rows
        for step in range(plan.P):
            tasks = [(t["q_off"], t["q_len"], t["k_off"], t["k_len"], t["causal"])
                     for t in plan.order if t["step"] == step]
            _lib.attn_bwd_group(qz, kz, vz, lse, delta, doz, dq_tiles, dk32, dv32, tasks, scale,
                                accumulate=step > 0)
    else:
        for t in plan.order:
            qs = slice(t["q_off"], t["q_off"] + t["q_len"])
            ks = slice(t["k_off"], t["k_off"] + t["k_len"])
            _lib.attn_bwd_ex(qz[:, qs], kz[:, ks], vz[:, ks], lse[:, :, qs], delta[:, :, qs], doz[:, qs],
                             dq32[:, qs], dk32[:, ks], dv32[:, ks], bool(t["causal"]), scale,
                             accumulate=t["step"] > 0)
    if fused:
        _lib.dq_untile(dq_tiles, grads[0])
    else:
        _lib.cast_f32_bf16(dq32, grads[0])
    for g32, g in zip(grads32[1:], grads[1:]):
        _lib.cast_f32_bf16(g32, g)
    return grads
