"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: their memory manager owns
all device memory, their memory plan is fixed at start-up, or they must not
call cudaMalloc because it can synchronise the device. attn_bwd_noalloc keeps
the Delta scratch in a fixed array inside the library instead; the array is
shared by every call on a device and keeps the last call's contents.

The test first fills the array with NaN (a call whose dO is +inf makes every
Delta it writes NaN, over more rows than the checked calls use), then calls
the entry point through the C ABI twice in a row. Each result must be finite,
so no Delta row was read before being rewritten, and must agree with
attn_bwd (caller-owned workspace) within the bf16 parity bars used by every
GPU test; the first also agrees with the fp64 oracle within the same bars.
It lives in its own file, collected last, and passes alone or after the rest.
"""

import ctypes

import pytest
import torch

import oracle
import long_context_causal_blockwise_gb300 as lcb
from long_context_causal_blockwise_gb300 import _lib
from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo
from parity import assert_bf16_close, to64

D = 128


def _poison_scratch(rows_needed):
    """One call whose Delta values are all NaN, over at least rows_needed (b, h, row) entries."""
    H, S = 8, 2048
    assert H * S >= rows_needed
    q, k, v, do = gaussian_qkvdo(1, H, S, D, seed=7)
    o, lse = lcb.attn_fwd(q, k, v, causal=True)
    do = torch.full_like(do, float("inf"))
    dq, dk, dv = lcb.attn_bwd_noalloc(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert torch.isnan(dq.float()).any()  # the poisoned Delta reached the gradients


@pytest.mark.gpu
def test_no_alloc_backward_twice_after_poisoned_scratch():
    cases = [(1, 4, 1024, True, 0), (2, 3, 777, False, 1)]
    _poison_scratch(max(B * H * S for B, H, S, _, _ in cases))
    for n, (B, H, S, causal, seed) in enumerate(cases):
        q, k, v, do = gaussian_qkvdo(B, H, S, D, seed=seed)
        o, lse = lcb.attn_fwd(q, k, v, causal=causal)
        ref = lcb.attn_bwd(q, k, v, o, lse, do, causal=causal)
        got = lcb.attn_bwd_noalloc(q, k, v, o, lse, do, causal=causal)
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(g.float()).all(), f"no-alloc {name}: non-finite (stale scratch read)"
            assert_bf16_close(to64(g), to64(r), f"no-alloc {name} vs attn_bwd B{B} H{H} S{S}")
        if n == 0:
            want = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, D ** -0.5)
            for name, g in zip(("dq", "dk", "dv"), got):
                assert_bf16_close(to64(g), want[name], f"no-alloc {name} vs oracle B{B} H{H} S{S}")


@pytest.mark.gpu
def test_no_alloc_rejects_oversized_problems():
    lib = _lib.load()
    limit = lib.attn_bwd_noalloc_max_rows()
    assert limit == 1 << 21
    nul = ctypes.c_void_p(0)
    rc = lib.attn_bwd_noalloc(nul, nul, nul, nul, nul, nul, nul, nul, nul, 1, 64, 32769, D, 1, 0.088, nul)
    assert rc == _lib.LCB_ERR_SCRATCH
    assert b"scratch" in lib.attn_status_string(rc)
