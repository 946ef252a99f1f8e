"""The oracle: a plain, slow, obviously correct fp64 CPU statement of what the
blockwise causal attention path computes.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and its ``--impl reference`` arm) may
import or call anything in this package. The product path (the CUDA library
and its Python binding) never imports it and never falls back to it.

The oracle shares no code with the CUDA path: no kernels, headers, helpers,
tables or constants. It reads the same bf16 input values (upcast to fp64) that
the CUDA path reads; nothing it returns ever comes from the CUDA path.

Sources (the web pages on EasyContext, cited by title and section):
  * "EasyContext核心技术解析：序列并行与Flash Attention的完美结合",
    §2 "Flash Attention优化": attention is computed exactly, tiled and with
    recomputation, never storing the full score matrix. Tiling and
    recomputation change only the order of the arithmetic, so the oracle is
    the textbook definition written out, with the full matrix materialised.
  * "EasyContext：用最少资源扩展大模型至百万Token": training uses full
    attention over the full sequence (no sparse or approximate attention).
  * "EasyContext代码解析200行核心训练脚本实现原理", §模型并行策略解析 and
    §训练循环核心逻辑: zigzag ring attention and the per-rank sequence split
    (prepare_seq_parallel_inputs).
  * "EasyContext核心技术解析…", §1 "序列并行技术": ring attention, whose ring
    steps compose by merging partial results over disjoint key sets.
  * "EasyContext核心技术解析…", §1 "序列并行技术": Ulysses attention, the
    sequence <-> head all-to-all around per-head attention (ulysses.py).
  * "EasyContext核心技术解析…", §3 "RoPE扩展技术": the raised rotary base
    (rope.py).
  * "EasyContext内存优化秘籍DeepSpeed Zero3卸载策略详解", §进阶优化与其他技术结合:
    the fused cross-entropy loss with an in-place backward (cross_entropy.py).

Parity pins: every function here is pinned by ``tests/test_oracle.py`` against
brute force, closed forms, invariants or finite differences; none is
"parity unpinned".
"""

from .attention import (  # noqa: F401
    attn_fwd,
    attn_probs,
    attn_bwd,
    attn_bwd_given_stats,
    attn_rows,
    attn_key_rows,
)
from .merge import lse_merge  # noqa: F401
from .rope import rope  # noqa: F401
from .cross_entropy import ce_fwd, ce_grad, ce_lse  # noqa: F401
from .ulysses import seq_to_head as ulysses_seq_to_head, head_to_seq as ulysses_head_to_seq  # noqa: F401
from .ulysses import ulysses_attn_fwd  # noqa: F401
from .zigzag import zigzag_schedule, zigzag_tasks_pairs, TASK_DIAG, TASK_LOWER, TASK_UPPER  # noqa: F401
from .zigzag import ring_schedule, TASK_FULL, TASK_NONE  # noqa: F401
