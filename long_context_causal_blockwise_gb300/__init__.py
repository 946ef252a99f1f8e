"""Blockwise causal attention for GB300 (sm_103a): the hot path of long-context
training with sequence parallelism, as a C-ABI CUDA library (libattn.so) with a
thin Python binding.

Public calls (all run in this library's CUDA kernels):
  attn_fwd, attn_fwd_ex, attn_fwd_group, attn_bwd, attn_bwd_ex, attn_bwd_group, attn_bwd_preprocess, attn_bwd_noalloc,
  dq_tiles_zeros / dq_tiles_zero_ / dq_untile (the one-pass backward's tiled dQ accumulator),
  attn_lse_merge, zigzag_schedule, ring_schedule, permute_rows, cast_f32_bf16,
  rope (rotary position embedding with a raised base, and its inverse),
  cross_entropy (the loss head with an in-place backward),
  zigzag_attention_fwd / zigzag_attention_bwd (the one-device zigzag ring),
  ulysses_all_to_all, ulysses_attention_fwd / ulysses_attention_bwd (Ulysses
  sequence parallelism over P ranks emulated on one device),
  RingRank / DistRingTransport / LoopbackRing (the rank-local zigzag ring
  driver: torch.distributed point-to-point between processes, or P ranks in
  one process).

The shared library is loaded on first use; importing the package does not
touch the GPU.
"""

from ._lib import (  # noqa: F401
    AttnError,
    attn_bwd,
    attn_bwd_ex,
    attn_bwd_group,
    attn_bwd_noalloc,
    attn_bwd_noalloc_max_rows,
    attn_bwd_preprocess,
    attn_bwd_workspace_bytes,
    attn_fwd,
    attn_fwd_ex,
    attn_fwd_group,
    attn_lse_merge,
    cast_f32_bf16,
    cross_entropy,
    dq_tiles_zero_,
    dq_tiles_zeros,
    dq_untile,
    load,
    permute_rows,
    ring_schedule,
    rope,
    selftest_bounded_wait,
    set_wait_limit_ns,
    take_device_status,
    ulysses_all_to_all,
    zigzag_schedule,
)
from .ring import DistRingTransport, LoopbackRing, RingRank, run_rank  # noqa: F401
from .ulysses import ulysses_attention_bwd, ulysses_attention_fwd  # noqa: F401
from .zigzag import zigzag_attention_bwd, zigzag_attention_fwd  # noqa: F401
