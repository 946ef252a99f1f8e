"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: their memory manager owns
all device memory, their memory plan is fixed at start-up, or they must not
call cudaMalloc because it can synchronise the device. attn_bwd_noalloc keeps
the Delta scratch in a fixed array inside the library instead. This test calls
it through the C ABI twice in a row (the array keeps the first call's contents
when the second starts) and checks each result against attn_bwd with a
caller-owned workspace, within the bf16 parity bars used by every GPU test.
It lives in its own file, collected last, and passes alone or after the rest.
"""

import ctypes

import pytest
import torch

import long_context_causal_blockwise_gb300 as lcb
from long_context_causal_blockwise_gb300 import _lib
from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo
from parity import assert_bf16_close, to64

D = 128


@pytest.mark.gpu
def test_no_alloc_backward_matches_workspace_backward_twice():
    cases = [(1, 4, 1024, True, 0), (2, 3, 777, False, 1)]
    for B, H, S, causal, seed in cases:
        q, k, v, do = gaussian_qkvdo(B, H, S, D, seed=seed)
        o, lse = lcb.attn_fwd(q, k, v, causal=causal)
        ref = lcb.attn_bwd(q, k, v, o, lse, do, causal=causal)
        got = lcb.attn_bwd_noalloc(q, k, v, o, lse, do, causal=causal)
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert_bf16_close(to64(g), to64(r), f"no-alloc {name} B{B} H{H} S{S}")


@pytest.mark.gpu
def test_no_alloc_rejects_oversized_problems():
    lib = _lib.load()
    limit = lib.attn_bwd_noalloc_max_rows()
    assert limit == 1 << 21
    nul = ctypes.c_void_p(0)
    rc = lib.attn_bwd_noalloc(nul, nul, nul, nul, nul, nul, nul, nul, nul, 1, 64, 32769, D, 1, 0.088, nul)
    assert rc == _lib.LCB_ERR_SCRATCH
    assert b"scratch" in lib.attn_status_string(rc)
