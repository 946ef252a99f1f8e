"""The C-ABI library builds, loads and exports every declared symbol; host-side
logic (argument checks, the zigzag schedule) works without a GPU."""

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from long_context_causal_blockwise_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lcb_attn.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"#.*", "", text)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\([^;{}]*\)\s*;", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("attn_fwd", "attn_bwd", "attn_lse_merge", "zigzag_schedule", "attn_fwd_ex", "attn_bwd_ex",
                 "attn_bwd_workspace_bytes", "attn_bwd_preprocess"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in _declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in _declared_functions():
        assert hasattr(lib, n)
    # the binding covers exactly what the header declares
    assert sorted(_lib.EXPORTED) == _declared_functions()


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.attn_status_string(code)
    assert lib.lcb_version() >= 100


def test_argument_errors_need_no_gpu(lib):
    nul = ctypes.c_void_p(0)
    # D != 128 is unsupported; checked before any CUDA call
    assert lib.attn_fwd(nul, nul, nul, nul, nul, 1, 1, 16, 64, 1, 0.1, nul) == _lib.LCB_ERR_UNSUPPORTED
    # bad sizes and null pointers
    assert lib.attn_fwd(nul, nul, nul, nul, nul, 0, 1, 16, 128, 1, 0.1, nul) == _lib.LCB_ERR_ARG
    assert lib.attn_fwd(nul, nul, nul, nul, nul, 1, 1, 16, 128, 1, 0.1, nul) == _lib.LCB_ERR_ARG
    assert lib.attn_fwd(nul, nul, nul, nul, nul, 1, 1, 16, 128, 2, 0.1, nul) == _lib.LCB_ERR_ARG
    assert lib.attn_fwd(nul, nul, nul, nul, nul, 1, 1, 16, 128, 1, -1.0, nul) == _lib.LCB_ERR_ARG
    # causal with Sq != Sk is unsupported
    assert lib.attn_fwd_ex(nul, nul, nul, nul, nul, 1, 1, 16, 32, 128, 1, 0.1, 128, 2048, 128, 4096, 128, 2048,
                           0, 16, 16, nul) == _lib.LCB_ERR_UNSUPPORTED
    # misaligned output pointer
    assert lib.attn_fwd_ex(nul, nul, nul, ctypes.c_void_p(8), ctypes.c_void_p(64), 1, 1, 16, 16, 128, 1, 0.1, 128,
                           2048, 128, 2048, 128, 2048, 0, 16, 16, nul) == _lib.LCB_ERR_ARG
    # empty problems are no-ops
    assert lib.attn_fwd(nul, nul, nul, nul, nul, 1, 1, 0, 128, 1, 0.1, nul) == _lib.LCB_OK
    assert lib.attn_lse_merge(nul, nul, nul, nul, 0, nul, 1, 1, 0, 128, 128, 0, 128, 0, 0, 0, 0, 0, nul) == _lib.LCB_OK
    assert lib.attn_lse_merge(nul, nul, nul, nul, 7, nul, 1, 1, 4, 128, 128, 0, 128, 0, 0, 0, 0, 0,
                              nul) == _lib.LCB_ERR_UNSUPPORTED
    assert lib.attn_bwd_workspace_bytes(2, 3, 100, 128) >= 2 * 3 * 100 * 4
    assert lib.attn_bwd(nul, nul, nul, nul, nul, nul, nul, nul, nul, 1, 1, 16, 128, 1, 0.1, nul, 0,
                        nul) == _lib.LCB_ERR_ARG
    assert lib.lcb_permute_rows(nul, nul, nul, 4, 24, nul) == _lib.LCB_ERR_ARG
    assert lib.lcb_cast_f32_bf16(nul, nul, -1, nul) == _lib.LCB_ERR_ARG


def test_fwd_group_argument_errors_need_no_gpu(lib):
    """attn_fwd_group rejects bad task tables before any CUDA call."""
    nul = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: every call below fails validation first

    def call(tasks, q_rows=1024, k_rows=1024, n=None):
        arr = (_lib.LcbFwdTask * max(1, len(tasks)))(*[_lib.LcbFwdTask(*t) for t in tasks])
        return lib.attn_fwd_group(fake, fake, fake, fake, fake, 1, 2, q_rows, k_rows, 128, 0.1, 256, 0, 256, 0, 256,
                                  0, 1024, 2048, arr, len(tasks) if n is None else n, nul)
    F32, BF16, MERGE = _lib.LCB_DTYPE_F32, _lib.LCB_DTYPE_BF16, _lib.LCB_OUT_F32_MERGE
    assert call([(0, 512, 0, 512, 0, F32), (256, 512, 0, 512, 0, F32)]) == _lib.LCB_ERR_ARG  # query rows overlap
    assert call([(0, 512, 600, 512, 0, F32)]) == _lib.LCB_ERR_ARG                            # keys past k_rows
    assert call([(-1, 16, 0, 16, 0, F32)]) == _lib.LCB_ERR_ARG                               # negative offset
    assert call([(0, 256, 0, 256, 0, F32), (256, 256, 0, 256, 0, BF16)]) == _lib.LCB_ERR_ARG  # one output dtype
    assert call([(0, 256, 0, 512, 1, MERGE)]) == _lib.LCB_ERR_UNSUPPORTED                    # causal needs a square
    assert call([(0, 256, 0, 256, 0, 9)]) == _lib.LCB_ERR_UNSUPPORTED                        # unknown output
    assert call([(0, 16, 0, 16, 0, F32)], n=17) == _lib.LCB_ERR_ARG                          # at most 16 tasks
    assert call([]) == _lib.LCB_OK                                                           # nothing to do


def test_bwd_group_rope_ce_argument_errors_need_no_gpu(lib):
    """The newer entry points reject bad arguments before any CUDA call."""
    nul = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)

    def bwd(tasks, n=None, tile_hs=16384 * 8):
        arr = (_lib.LcbBwdTask * max(1, len(tasks)))(*[_lib.LcbBwdTask(*t) for t in tasks])
        return lib.attn_bwd_fused_group(fake, fake, fake, fake, fake, fake, fake, fake, fake, 1, 2, 1024, 1024, 128,
                                        0.1, 256, 0, 256, 0, 1024, 2048, _lib.LCB_GRAD_BF16, tile_hs, 0, 256, 0, arr,
                                        len(tasks) if n is None else n, nul)
    assert bwd([(64, 128, 0, 128, 0)]) == _lib.LCB_ERR_ARG                             # q_off not on a dQ tile
    assert bwd([(0, 128, 0, 256, 0), (128, 128, 128, 256, 0)]) == _lib.LCB_ERR_ARG     # key ranges overlap
    assert bwd([(0, 128, 900, 256, 0)]) == _lib.LCB_ERR_ARG                            # keys past k_rows
    assert bwd([(0, 128, 0, 256, 1)]) == _lib.LCB_ERR_UNSUPPORTED                      # causal needs a square
    assert bwd([(0, 128, 0, 128, 0)], tile_hs=3) == _lib.LCB_ERR_ARG                   # tile stride not 16-byte
    assert bwd([(0, 128, 0, 128, 0)], n=17) == _lib.LCB_ERR_ARG                        # at most 16 tasks
    # RoPE: D, theta, inverse flag, alignment, row stride
    assert lib.lcb_rope(fake, fake, 1, 8, 2, 64, 1e6, 0, 0, 256, 0, nul) == _lib.LCB_ERR_UNSUPPORTED
    assert lib.lcb_rope(fake, fake, 1, 8, 2, 128, -1.0, 0, 0, 256, 0, nul) == _lib.LCB_ERR_ARG
    assert lib.lcb_rope(fake, fake, 1, 8, 2, 128, 1e6, 0, 2, 256, 0, nul) == _lib.LCB_ERR_ARG
    assert lib.lcb_rope(ctypes.c_void_p(2), fake, 1, 8, 2, 128, 1e6, 0, 0, 256, 0, nul) == _lib.LCB_ERR_ARG
    assert lib.lcb_rope(fake, fake, 1, 8, 2, 128, 1e6, 0, 0, 128, 0, nul) == _lib.LCB_ERR_ARG
    assert lib.lcb_rope(fake, fake, 1, 0, 2, 128, 1e6, 0, 0, 256, 0, nul) == _lib.LCB_OK
    # cross-entropy: mode, row stride, empty vocabulary, null pointers, empty
    assert lib.lcb_cross_entropy(fake, fake, fake, fake, nul, 4, 100, 100, -100, 3, nul) == _lib.LCB_ERR_UNSUPPORTED
    assert lib.lcb_cross_entropy(fake, fake, fake, fake, nul, 4, 100, 99, -100, 0, nul) == _lib.LCB_ERR_ARG
    assert lib.lcb_cross_entropy(fake, fake, fake, fake, nul, 4, 0, 100, -100, 0, nul) == _lib.LCB_ERR_ARG
    assert lib.lcb_cross_entropy(fake, nul, fake, fake, nul, 4, 100, 100, -100, 1, nul) == _lib.LCB_ERR_ARG
    assert lib.lcb_cross_entropy(fake, fake, fake, fake, nul, 0, 100, 100, -100, 1, nul) == _lib.LCB_OK
    # dQ accumulator helpers
    assert lib.lcb_dq_untile(fake, 3, 0, fake, 256, 0, 1, 2, 16, nul) == _lib.LCB_ERR_ARG
    assert lib.lcb_dq_tiles_zero(ctypes.c_void_p(4), 16, nul) == _lib.LCB_ERR_ARG
    assert lib.attn_bwd_workspace_bytes(1, 2, 300, 128) == 2 * 300 * 4 + 1 * 2 * 3 * 16384 * 4 + 256 - (2 * 300 * 4) % 256


@pytest.mark.parametrize("S,P", [(8, 2), (16, 1), (48, 3), (256, 4), (256, 8), (131072, 8), (524288, 8)])
def test_zigzag_schedule_matches_oracle_bit_exact(lib, S, P):
    perm, tasks = _lib.zigzag_schedule(S, P)
    operm, otasks = oracle.zigzag_schedule(S, P)
    assert np.array_equal(np.array(perm), operm)
    assert tasks == otasks


@pytest.mark.parametrize("S,P", [(6, 3), (8, 1), (4096, 8), (131072, 8), (100, 5)])
def test_ring_schedule_matches_oracle_bit_exact(lib, S, P):
    perm, tasks = _lib.ring_schedule(S, P)
    operm, otasks = oracle.ring_schedule(S, P)
    assert np.array_equal(np.array(perm), operm)
    assert tasks == otasks


def test_ring_schedule_rejects_bad_sizes(lib):
    nul = ctypes.POINTER(ctypes.c_int)()
    for S, P in ((7, 2), (0, 1), (4, 0), (3, 4)):
        assert lib.ring_schedule(S, P, nul, None) == _lib.LCB_ERR_SCHEDULE


def test_zigzag_schedule_rejects_bad_sizes(lib):
    for S, P in ((10, 3), (0, 1), (8, 0), (3, 2), (-8, 2)):
        assert lib.zigzag_schedule(S, P, None, None) == _lib.LCB_ERR_SCHEDULE
    with pytest.raises(_lib.AttnError) as e:
        _lib.zigzag_schedule(10, 3)
    assert e.value.status == _lib.LCB_ERR_SCHEDULE


def test_zigzag_c3_tile_counts_match_monolithic():
    """At S = 131072, P = 8 the tasks cover as many 128x128 causal tiles as monolithic attention."""
    S, P, T = 131072, 8, 128
    perm, tasks = _lib.zigzag_schedule(S, P)
    n = S // T
    mono_pairs = S * (S + 1) // 2
    mono_tiles = n * (n + 1) // 2
    pairs = tiles = 0
    for t in tasks:
        a, b = t["q_len"] // T, t["k_len"] // T
        if t["causal"]:
            pairs += t["q_len"] * (t["q_len"] + 1) // 2
            tiles += a * (a + 1) // 2
        else:
            pairs += t["q_len"] * t["k_len"]
            tiles += a * b
    assert pairs == mono_pairs
    assert tiles == mono_tiles
