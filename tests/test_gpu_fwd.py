"""GPU parity of the forward kernel, the LSE merge, the preprocess and the
permutation kernels against the fp64 oracle, through the C ABI."""

import math

import numpy as np
import pytest
import torch

import oracle
import long_context_causal_blockwise_gb300 as lcb
from long_context_causal_blockwise_gb300 import _lib
from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo, sample_rows
from parity import assert_bf16_close, assert_lse_close, to64

pytestmark = pytest.mark.gpu
D = 128


def _fwd_check(B, H, S, causal, seed, scale=None):
    q, k, v, _ = gaussian_qkvdo(B, H, S, D, seed=seed, with_do=False)
    scale = D ** -0.5 if scale is None else scale
    o, lse = lcb.attn_fwd(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    O, L = oracle.attn_fwd(to64(q), to64(k), to64(v), causal, scale)
    assert_bf16_close(to64(o), O, f"O B{B} H{H} S{S} causal{causal}")
    assert_lse_close(to64(lse), L)
    return q, k, v, o, lse


def test_config1_full_tensors():
    """B=1, H=4, S=1024, D=128, causal: every output against the oracle."""
    _fwd_check(1, 4, 1024, True, seed=0)


@pytest.mark.parametrize("S", [1, 7, 128, 129, 255, 256, 257, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_lengths(S, causal):
    _fwd_check(2, 3, S, causal, seed=S)


def test_first_row_is_exactly_v0():
    """Causal row 0 has one visible key: weight exactly 1, so O[:,0] == V[:,0] bit for bit."""
    q, k, v, o, lse = _fwd_check(1, 4, 640, True, seed=3)
    assert torch.equal(o[:, 0], v[:, 0])
    want = (q[:, 0].double() * k[:, 0].double()).sum(-1) * D ** -0.5  # [B, H]
    np.testing.assert_allclose(lse[:, :, 0].double().cpu().numpy(), want.cpu().numpy(), atol=1e-3)


def test_peaked_scores_large_magnitude():
    """Scores near 1e3 with a lead of > 40 on the latest key: online max must hold."""
    B, H, S = 1, 2, 384
    v = torch.randn(B, S, H, D, device="cuda").to(torch.bfloat16)
    k = torch.zeros(B, S, H, D, device="cuda")
    k[..., 0] = torch.arange(S, device="cuda", dtype=torch.float32)[None, :, None] / 8.0
    q = torch.zeros(B, S, H, D, device="cuda")
    q[..., 0] = 512.0
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    o, lse = lcb.attn_fwd(q, k, v, causal=True, scale=1.0)
    torch.cuda.synchronize()
    O, L = oracle.attn_fwd(to64(q), to64(k), to64(v), True, 1.0)
    assert_bf16_close(to64(o), O, "O peaked")
    np.testing.assert_allclose(to64(lse), L, rtol=1e-6, atol=1e-3)


def test_rectangular_noncausal_and_fp32_output():
    B, H, Sq, Sk = 1, 2, 300, 517
    g = torch.Generator(device="cuda").manual_seed(11)
    q = torch.randn(B, Sq, H, D, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, Sk, H, D, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, Sk, H, D, generator=g, device="cuda").to(torch.bfloat16)
    o = torch.empty(B, Sq, H, D, dtype=torch.float32, device="cuda")
    lse = torch.empty(B, H, Sq, dtype=torch.float32, device="cuda")
    lcb.attn_fwd_ex(q, k, v, o, lse, False, D ** -0.5)
    torch.cuda.synchronize()
    O, L = oracle.attn_fwd(to64(q), to64(k), to64(v), False, D ** -0.5)
    assert_bf16_close(to64(o), O, "O fp32 out", max_abs=5e-3, mean_abs=5e-4)
    assert_lse_close(to64(lse), L)


def test_strided_subranges_like_ring_steps():
    """Row windows of larger tensors, as the zigzag ring addresses its chunks."""
    B, H, S = 1, 2, 1024
    q, k, v, _ = gaussian_qkvdo(B, H, S, D, seed=5, with_do=False)
    o = torch.zeros(B, S, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, H, S, dtype=torch.float32, device="cuda")
    qs, ks = slice(512, 768), slice(128, 384)
    lcb.attn_fwd_ex(q[:, qs], k[:, ks], v[:, ks], o[:, qs], lse[:, :, qs], False, D ** -0.5)
    lcb.attn_fwd_ex(q[:, 0:256], k[:, 0:256], v[:, 0:256], o[:, 0:256], lse[:, :, 0:256], True, D ** -0.5)
    torch.cuda.synchronize()
    O1, L1 = oracle.attn_fwd(to64(q[:, qs]), to64(k[:, ks]), to64(v[:, ks]), False, D ** -0.5)
    O2, L2 = oracle.attn_fwd(to64(q[:, :256]), to64(k[:, :256]), to64(v[:, :256]), True, D ** -0.5)
    assert_bf16_close(to64(o[:, qs]), O1, "O window")
    assert_lse_close(to64(lse[:, :, qs]), L1)
    assert_bf16_close(to64(o[:, :256]), O2, "O causal window")
    assert_lse_close(to64(lse[:, :, :256]), L2)
    # rows outside the windows were not touched
    assert torch.count_nonzero(o[:, 256:512]) == 0 and torch.count_nonzero(o[:, 768:]) == 0


def test_empty_key_set():
    B, H, Sq = 1, 2, 10
    q = torch.randn(B, Sq, H, D, device="cuda").to(torch.bfloat16)
    kv = torch.empty(B, 0, H, D, device="cuda", dtype=torch.bfloat16)
    o = torch.full((B, Sq, H, D), 7.0, device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros(B, H, Sq, device="cuda")
    lcb.attn_fwd_ex(q, kv, kv, o, lse, False, D ** -0.5)
    torch.cuda.synchronize()
    assert torch.count_nonzero(o) == 0
    assert torch.isneginf(lse).all()


def test_lse_merge_matches_oracle_and_split_equals_monolithic():
    B, H, Sq, Sk = 1, 4, 384, 1024
    g = torch.Generator(device="cuda").manual_seed(21)
    q = torch.randn(B, Sq, H, D, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, Sk, H, D, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, Sk, H, D, generator=g, device="cuda").to(torch.bfloat16)
    o_acc = torch.empty(B, Sq, H, D, dtype=torch.float32, device="cuda")
    lse_acc = torch.empty(B, H, Sq, dtype=torch.float32, device="cuda")
    o_b = torch.empty(B, Sq, H, D, dtype=torch.bfloat16, device="cuda")
    lse_b = torch.empty(B, H, Sq, dtype=torch.float32, device="cuda")
    o_out = torch.empty(B, Sq, H, D, dtype=torch.bfloat16, device="cuda")
    lcb.attn_fwd_ex(q, k[:, :400], v[:, :400], o_acc, lse_acc, False, D ** -0.5)
    lcb.attn_fwd_ex(q, k[:, 400:], v[:, 400:], o_b, lse_b, False, D ** -0.5)
    oa, la, ob, lb = to64(o_acc), to64(lse_acc), to64(o_b), to64(lse_b)
    lcb.attn_lse_merge(o_acc, lse_acc, o_b, lse_b, o_out_bf16=o_out)
    torch.cuda.synchronize()
    Om, Lm = oracle.lse_merge(oa, la, ob, lb)
    np.testing.assert_allclose(to64(o_acc), Om, atol=1e-5)
    np.testing.assert_allclose(to64(lse_acc), Lm, atol=1e-5)
    O, L = oracle.attn_fwd(to64(q), to64(k), to64(v), False, D ** -0.5)
    assert_bf16_close(to64(o_out), O, "merged O")
    assert_lse_close(to64(lse_acc), L)


@pytest.mark.parametrize("B,H", [(1, 2), (2, 6)])
def test_lse_merge_empty_sides(B, H):
    """Both merge kernels (a warp per (row, head) for H < 4, a warp per row over
    the heads otherwise, here with a partial group of heads)."""
    R = 64
    o_acc = torch.randn(B, R, H, D, device="cuda")
    lse_acc = torch.randn(B, H, R, device="cuda")
    lse_acc[:, :, ::3] = -math.inf
    o_acc[:, ::3] = 0
    o_b = torch.randn(B, R, H, D, device="cuda")
    lse_b = torch.full((B, H, R), -math.inf, device="cuda")
    lse_b[:, :, 1::3] = 0.25
    want = oracle.lse_merge(to64(o_acc), to64(lse_acc), to64(o_b), to64(lse_b))
    lcb.attn_lse_merge(o_acc, lse_acc, o_b, lse_b)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to64(o_acc), want[0], atol=1e-5)
    got_l = to64(lse_acc)
    assert np.array_equal(np.isneginf(got_l), np.isneginf(want[1]))
    fin = np.isfinite(want[1])
    np.testing.assert_allclose(got_l[fin], want[1][fin], atol=1e-5)


@pytest.mark.parametrize("ob_f32,with_out", [(False, False), (False, True), (True, False), (True, True)])
def test_lse_merge_rows_kernel_all_forms(ob_f32, with_out):
    """The row kernel's four forms (block result bf16 or fp32, with or without
    the bf16 copy out), B = 2 and H = 12 (a group of eight heads and a partial
    one), against the oracle; the copy out is the merged fp32 value rounded
    once."""
    B, H, R = 2, 12, 200
    g = torch.Generator(device="cuda").manual_seed(5 + 2 * ob_f32 + with_out)
    o_acc = torch.randn(B, R, H, D, generator=g, device="cuda")
    lse_acc = torch.randn(B, H, R, generator=g, device="cuda") * 4
    lse_acc[:, :, ::5] = -math.inf
    o_b = torch.randn(B, R, H, D, generator=g, device="cuda")
    o_b = o_b if ob_f32 else o_b.to(torch.bfloat16)
    lse_b = torch.randn(B, H, R, generator=g, device="cuda") * 4
    lse_b[:, :, ::7] = -math.inf
    want = oracle.lse_merge(to64(o_acc), to64(lse_acc), to64(o_b), to64(lse_b))
    o_out = torch.empty(B, R, H, D, dtype=torch.bfloat16, device="cuda") if with_out else None
    lcb.attn_lse_merge(o_acc, lse_acc, o_b, lse_b, o_out_bf16=o_out)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to64(o_acc), want[0], atol=1e-5)
    got_l = to64(lse_acc)
    assert np.array_equal(np.isneginf(got_l), np.isneginf(want[1]))
    fin = np.isfinite(want[1])
    np.testing.assert_allclose(got_l[fin], want[1][fin], atol=1e-5)
    if with_out:
        assert torch.equal(o_out, o_acc.to(torch.bfloat16))


@pytest.mark.parametrize("H", [3, 4, 10])
def test_preprocess_delta(H):
    """Both preprocess kernels (odd H: a warp per (row, head); even H: a warp per row)."""
    B, S = 2, 777
    o, do, _, _ = gaussian_qkvdo(B, H, S, D, seed=9, with_do=False)
    delta = torch.empty(B, H, S, device="cuda")
    lcb.attn_bwd_preprocess(o, do, delta)
    torch.cuda.synchronize()
    want = np.einsum("bshd,bshd->bhs", to64(o), to64(do))
    np.testing.assert_allclose(to64(delta), want, atol=1e-3, rtol=1e-5)


def test_zigzag_gather_scatter_bit_exact():
    S, P, H = 4096, 4, 2
    x = torch.randn(1, S, H, D, device="cuda").to(torch.bfloat16)
    plan = lcb.zigzag.ZigzagPlan(S, P, "cuda")
    perm, _ = oracle.zigzag_schedule(S, P)
    xz = plan.gather(x)
    assert torch.equal(xz, x[:, torch.as_tensor(perm, device="cuda")])
    assert torch.equal(plan.scatter(xz), x)


def test_bounded_wait_expires_and_context_survives():
    old = lcb.set_wait_limit_ns(50_000_000)  # 50 ms
    try:
        assert lcb.selftest_bounded_wait() == _lib.LCB_ERR_TIMEOUT
    finally:
        lcb.set_wait_limit_ns(old)
    assert lcb.take_device_status()[0] == 0
    _fwd_check(1, 1, 256, True, seed=1)


def test_config2_sampled_rows_forward():
    """B=1, H=32, S=32768 (Llama-2-7B layer): sampled query rows on every head."""
    B, H, S = 1, 32, 32768
    q, k, v, _ = gaussian_qkvdo(B, H, S, D, seed=0, with_do=False)
    o, lse = lcb.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    rows = sample_rows(S, 256, seed=0)
    ref = oracle.attn_rows(to64(q), to64(k), to64(v), None, rows, True, D ** -0.5)
    assert_bf16_close(to64(o[:, rows]), ref["o"], "O C2 sampled")
    assert_lse_close(to64(lse[:, :, rows]), ref["lse"])


def test_grouped_launch_equals_separate_calls():
    """attn_fwd_group runs several blocks in one launch: every output equals
    the attn_fwd_ex call of the same block bit for bit, for causal and
    rectangular blocks, ragged lengths, fp32 store and merge outputs, and
    blocks without keys (store: O = 0, LSE = -inf; merge: untouched)."""
    B, H, S = 2, 3, 1500
    g = torch.Generator(device="cuda").manual_seed(31)
    q, k, v = (torch.randn(B, S, H, D, generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    scale = D ** -0.5
    tasks = [(0, 300, 0, 300, 1, "f32"),       # causal diagonal block
             (300, 256, 700, 513, 0, "f32"),   # rectangular, ragged keys
             (556, 129, 0, 1500, 0, "merge"),  # merge into an accumulator, ragged queries
             (685, 400, 100, 200, 0, "merge"),
             (1085, 77, 0, 0, 0, "f32"),       # no keys: stored as empty
             (1162, 60, 0, 0, 0, "merge"),     # no keys: accumulator untouched
             (1222, 278, 1222, 278, 1, "f32")]
    acc0 = torch.randn(B, S, H, D, generator=g, device="cuda")
    lse0 = torch.randn(B, H, S, generator=g, device="cuda")
    o1, l1 = acc0.clone(), lse0.clone()
    lcb.attn_fwd_group(q, k, v, o1, l1, tasks, scale)
    o2, l2 = acc0.clone(), lse0.clone()
    for qo, ql, ko, kl, causal, out in tasks:
        qs, ks = slice(qo, qo + ql), slice(ko, ko + kl)
        lcb.attn_fwd_ex(q[:, qs], k[:, ks], v[:, ks], o2[:, qs], l2[:, :, qs], bool(causal), scale,
                        merge=(out == "merge"))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # and a store-mode block against the oracle
    ref_o, ref_l = oracle.attn_fwd(to64(q[:, 300:556]), to64(k[:, 700:1213]), to64(v[:, 700:1213]), False, scale)
    assert_bf16_close(to64(o1[:, 300:556]), ref_o, "O grouped block")
    assert_lse_close(to64(l1[:, :, 300:556]), ref_l)
    assert (o1[:, 1085:1162] == 0).all() and torch.isneginf(l1[:, :, 1085:1162]).all()
    assert torch.equal(o1[:, 1162:1222], acc0[:, 1162:1222])
