"""GPU parity of the backward passes (dK/dV and dQ) against the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
import long_context_causal_blockwise_gb300 as lcb
from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo, sample_rows
from parity import (assert_bf16_close, assert_bf16_close_scaled, assert_lse_close, err_stats, head64, map_heads, oracle_rows_by_head,
                    rows_budget, to64)

pytestmark = pytest.mark.gpu
D = 128


def _bwd_full_check(B, H, S, causal, seed):
    q, k, v, do = gaussian_qkvdo(B, H, S, D, seed=seed)
    o, lse = lcb.attn_fwd(q, k, v, causal=causal)
    dq, dk, dv = lcb.attn_bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    ref = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, D ** -0.5)
    tag = f"B{B} H{H} S{S} causal{causal}"
    assert_bf16_close(to64(dq), ref["dq"], "dQ " + tag)
    assert_bf16_close(to64(dk), ref["dk"], "dK " + tag)
    assert_bf16_close(to64(dv), ref["dv"], "dV " + tag)


def test_config1_shape_backward_full_tensors():
    _bwd_full_check(1, 4, 1024, True, seed=0)


@pytest.mark.parametrize("S", [1, 7, 128, 129, 256, 383, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_lengths(S, causal):
    _bwd_full_check(2, 2, S, causal, seed=100 + S)


def test_block_backward_accumulates_to_monolithic():
    """Key blocks with the full problem's LSE/Delta, fp32 accumulate, add up exactly."""
    B, H, Sq, Sk = 1, 2, 256, 640
    g = torch.Generator(device="cuda").manual_seed(3)
    mk = lambda n: torch.randn(B, n, H, D, generator=g, device="cuda").to(torch.bfloat16)  # noqa: E731
    q, k, v, do = mk(Sq), mk(Sk), mk(Sk), mk(Sq)
    o = torch.empty(B, Sq, H, D, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(B, H, Sq, device="cuda")
    lcb.attn_fwd_ex(q, k, v, o, lse, False, D ** -0.5)
    delta = torch.empty(B, H, Sq, device="cuda")
    lcb.attn_bwd_preprocess(o, do, delta)
    dq = torch.zeros(B, Sq, H, D, device="cuda")
    dk = torch.zeros(B, Sk, H, D, device="cuda")
    dv = torch.zeros(B, Sk, H, D, device="cuda")
    cuts = [(0, 200), (200, 456), (456, 640)]
    for a, b in cuts:
        # fp32 accumulate: dq sums over the blocks, each block adds to its own dk/dv rows
        lcb.attn_bwd_ex(q, k[:, a:b], v[:, a:b], lse, delta, do, dq, dk[:, a:b], dv[:, a:b], False, D ** -0.5,
                        accumulate=True)
    torch.cuda.synchronize()
    ref = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), False, D ** -0.5)
    assert_bf16_close(to64(dq), ref["dq"], "dQ blocks")
    assert_bf16_close(to64(dk), ref["dk"], "dK blocks")
    assert_bf16_close(to64(dv), ref["dv"], "dV blocks")
    # fp32 store mode overwrites: a second pass over one block in store mode equals that block alone
    dk2 = torch.full_like(dk[:, :200], 9.0)
    dv2 = torch.full_like(dv[:, :200], 9.0)
    dq2 = torch.full_like(dq, 9.0)
    lcb.attn_bwd_ex(q, k[:, :200], v[:, :200], lse, delta, do, dq2, dk2, dv2, False, D ** -0.5, accumulate=False)
    torch.cuda.synchronize()
    assert torch.equal(dk2, dk[:, :200]) and torch.equal(dv2, dv[:, :200])


def test_split_passes_match_combined():
    B, H, S = 1, 2, 512
    q, k, v, do = gaussian_qkvdo(B, H, S, D, seed=8)
    o, lse = lcb.attn_fwd(q, k, v)
    delta = torch.empty(B, H, S, device="cuda")
    lcb.attn_bwd_preprocess(o, do, delta)
    g1 = [torch.empty_like(q) for _ in range(3)]
    g2 = [torch.full_like(q, 3.0) for _ in range(3)]
    lcb.attn_bwd_ex(q, k, v, lse, delta, do, *g1, True, D ** -0.5)
    lcb.attn_bwd_ex(q, k, v, lse, delta, do, *g2, True, D ** -0.5, passes="dkdv")
    torch.cuda.synchronize()
    assert torch.equal(g2[1], g1[1]) and torch.equal(g2[2], g1[2])
    assert (g2[0] == 3.0).all()  # dq untouched by the dK/dV pass
    lcb.attn_bwd_ex(q, k, v, lse, delta, do, *g2, True, D ** -0.5, passes="dq")
    torch.cuda.synchronize()
    assert torch.equal(g2[0], g1[0])


def test_empty_sides():
    """Sk = 0: dQ is zero; Sq = 0: dK and dV are zero."""
    B, H = 1, 2
    q = torch.randn(B, 64, H, D, device="cuda").to(torch.bfloat16)
    e = torch.empty(B, 0, H, D, device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros(B, H, 64, device="cuda")
    delta = torch.zeros(B, H, 64, device="cuda")
    dq = torch.full_like(q, 5.0)
    lcb.attn_bwd_ex(q, e, e, lse, delta, q, dq, e, e, False, D ** -0.5)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dq) == 0
    dk = torch.full_like(q, 5.0)
    dv = torch.full_like(q, 5.0)
    le = torch.zeros(B, H, 0, device="cuda")
    lcb.attn_bwd_ex(e, q, q, le, le, e, e, dk, dv, False, D ** -0.5)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0


def test_config2_sampled_rows_backward():
    """B=1, H=32, S=32768: O, LSE and dQ on 4096 sampled query rows of every
    head; dK/dV on 4096 sampled key rows of two heads; the sum invariants on
    every head."""
    B, H, S = 1, 32, 32768
    scale = D ** -0.5
    q, k, v, do = gaussian_qkvdo(B, H, S, D, seed=0)
    o, lse = lcb.attn_fwd(q, k, v)
    dq, dk, dv = lcb.attn_bwd(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    rows = sample_rows(S, rows_budget(4096), seed=1)
    refs = oracle_rows_by_head(q, k, v, do, rows, True, scale)
    rows_d = torch.as_tensor(rows, device="cuda")
    assert_bf16_close(to64(o[:, rows_d]), np.concatenate([r["o"] for r in refs], 2), "O C2 sampled")
    assert_lse_close(to64(lse[:, :, rows_d]), np.concatenate([r["lse"] for r in refs], 1))
    assert_bf16_close(to64(dq[:, rows_d]), np.concatenate([r["dq"] for r in refs], 2), "dQ C2 sampled")
    keys = sample_rows(S, rows_budget(4096), seed=2)
    keys_d = torch.as_tensor(keys, device="cuda")
    heads = [0, 31]
    kref = map_heads(lambda h: oracle.attn_key_rows(*(head64(t, h) for t in (q, k, v, do)), keys, [0], True, scale),
                     heads)
    for h, (rdk, rdv) in zip(heads, kref):
        assert_bf16_close(to64(dk[:, keys_d, h:h + 1]), rdk, f"dK C2 sampled head {h}")
        assert_bf16_close(to64(dv[:, keys_d, h:h + 1]), rdv, f"dV C2 sampled head {h}")
    # sum_j dV_j = sum_i dO_i and sum_j dK_j = 0, per head (fp32 sums of bf16 values)
    sdv = dv.float().sum(1)
    sdo = do.float().sum(1)
    sdk = dk.float().sum(1)
    tol = 1e-2 * sdo.norm(dim=-1, keepdim=True)
    assert ((sdv - sdo).norm(dim=-1, keepdim=True) <= tol).all()
    assert (sdk.norm(dim=-1) <= 1e-2 * dk.float().norm(dim=(1, 3))).all()


def _stats(q, k, v, do, causal, scale):
    B, Sq, H, _ = q.shape
    o = torch.empty(B, Sq, H, D, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(B, H, Sq, device="cuda")
    lcb.attn_fwd_ex(q, k, v, o, lse, causal, scale)
    delta = torch.empty(B, H, Sq, device="cuda")
    lcb.attn_bwd_preprocess(o, do, delta)
    return lse, delta


def untile_f32(tiles, S):
    """The tiled dQ accumulator as fp32 [B, S, H, D]: columns 0-63 as two
    row-swizzled blocks, columns 64-127 chunk-major."""
    B, H, T, _ = tiles.shape
    t = tiles.view(B, H, T, 16384)
    lo = t[..., :8192].reshape(B, H, T, 2, 128, 8, 4)
    r = torch.arange(128, device=tiles.device)
    c = torch.arange(8, device=tiles.device)
    pos = c[None, :] ^ (r[:, None] & 7)
    g = lo[:, :, :, :, r[:, None], pos, :]  # [B, H, T, 2, 128, 8, 4]
    lo_rows = g.permute(0, 2, 4, 1, 3, 5, 6).reshape(B, T * 128, H, 64)
    hi = t[..., 8192:].reshape(B, H, T, 16, 128, 4)
    hi_rows = hi.permute(0, 2, 4, 1, 3, 5).reshape(B, T * 128, H, 64)
    return torch.cat([lo_rows, hi_rows], dim=3)[:, :S]


@pytest.mark.parametrize("B,H,Sq,Sk,causal", [(2, 3, 700, 700, True), (1, 2, 300, 520, False),
                                              (1, 2, 130, 70, False), (1, 1, 1, 1, True)])
def test_fused_pass_vs_two_pass_and_oracle(B, H, Sq, Sk, causal):
    """The one-pass backward: dK/dV bit-identical to the two-pass dK/dV pass
    (same products in the same order), dQ (bulk fp32 reductions into the tiled
    accumulator) within fp32 rounding of the two-pass dQ, and all three
    against the oracle; lcb_dq_untile gives the accumulator's bf16 rows."""
    scale = D ** -0.5
    g = torch.Generator(device="cuda").manual_seed(Sq * 7 + Sk)
    mk = lambda n: torch.randn(B, n, H, D, generator=g, device="cuda").to(torch.bfloat16)  # noqa: E731
    q, k, v, do = mk(Sq), mk(Sk), mk(Sk), mk(Sq)
    lse, delta = _stats(q, k, v, do, causal, scale)
    f32 = lambda n: torch.full((B, n, H, D), 7.0, device="cuda")  # noqa: E731
    tiles, dk1, dv1 = lcb.dq_tiles_zeros(B, H, Sq, "cuda"), f32(Sk), f32(Sk)
    lcb.attn_bwd_ex(q, k, v, lse, delta, do, tiles, dk1, dv1, causal, scale, accumulate=False, passes="fused")
    dq2, dk2, dv2 = f32(Sq), f32(Sk), f32(Sk)
    lcb.attn_bwd_ex(q, k, v, lse, delta, do, dq2, dk2, dv2, causal, scale, accumulate=False)
    dq16 = lcb.dq_untile(tiles, torch.empty_like(q))
    torch.cuda.synchronize()
    dq1 = untile_f32(tiles, Sq)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert torch.allclose(dq1, dq2, rtol=1e-4, atol=1e-5)
    assert torch.equal(dq16, dq1.to(torch.bfloat16))
    ref = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), causal, scale)
    assert_bf16_close(to64(dq1), ref["dq"], "dQ fused")
    assert_bf16_close(to64(dk1), ref["dk"], "dK fused")
    assert_bf16_close(to64(dv1), ref["dv"], "dV fused")


def test_fused_pass_adds_into_dq_and_masks_ragged_keys():
    """dQ is added into (two calls give twice one call), and a ragged key tile
    whose zero-filled rows would score exp(-LSE) = inf for very negative LSE
    leaves everything finite."""
    B, H, Sq, Sk = 1, 2, 160, 70
    scale = D ** -0.5
    k = torch.ones(B, Sk, H, D, device="cuda", dtype=torch.bfloat16)
    q = torch.full((B, Sq, H, D), -150.0 / (D * scale), device="cuda").to(torch.bfloat16)  # scores about -150
    g = torch.Generator(device="cuda").manual_seed(11)
    v = torch.randn(B, Sk, H, D, generator=g, device="cuda").to(torch.bfloat16)
    do = torch.randn(B, Sq, H, D, generator=g, device="cuda").to(torch.bfloat16)
    lse, delta = _stats(q, k, v, do, False, scale)
    assert (lse < -140).all()
    tiles = lcb.dq_tiles_zeros(B, H, Sq, "cuda")
    dk = torch.empty(B, Sk, H, D, device="cuda", dtype=torch.bfloat16)
    dv = torch.empty_like(dk)
    lcb.attn_bwd_ex(q, k, v, lse, delta, do, tiles, dk, dv, False, scale, passes="fused")
    once = untile_f32(tiles, Sq).clone()
    lcb.attn_bwd_ex(q, k, v, lse, delta, do, tiles, dk, dv, False, scale, passes="fused")
    torch.cuda.synchronize()
    twice = untile_f32(tiles, Sq)
    for t in (once, dk, dv):
        assert torch.isfinite(t).all()
    assert torch.allclose(twice, 2 * once, rtol=1e-6, atol=1e-6)
    # the two-pass form masks the ragged keys explicitly: same dK/dV bits, dQ within fp32 rounding
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(dk), torch.empty_like(dv)
    lcb.attn_bwd_ex(q, k, v, lse, delta, do, dq2, dk2, dv2, False, scale)
    torch.cuda.synchronize()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert torch.allclose(once.to(torch.bfloat16).float(), dq2.float(), rtol=2e-2, atol=1e-3)
    # against the oracle: |dK| is about 1 here, so relative L2 (bf16 rounding); dQ is 0 up to the rounding of dS
    ref = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), False, scale)
    for got, want, name in ((dk, ref["dk"], "dK"), (dv, ref["dv"], "dV")):
        _, _, rel = err_stats(to64(got), want)
        assert rel <= 1e-2, f"{name} fused, ragged keys: rel-L2 {rel:.3e}"
    assert np.abs(to64(once) - ref["dq"]).max() <= 2e-2


def test_monolithic_backward_two_calls_agree():
    """attn_bwd (fused; dQ partials added by bulk reductions in L2) is repeatable to within bf16
    rounding; dK and dV are bit-identical."""
    q, k, v, do = gaussian_qkvdo(1, 4, 1024, D, seed=21)
    o, lse = lcb.attn_fwd(q, k, v)
    g1 = lcb.attn_bwd(q, k, v, o, lse, do)
    g2 = lcb.attn_bwd(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert (g1[0].float() - g2[0].float()).abs().max().item() <= 2 ** -8 * g1[0].float().abs().max().item()


def test_grouped_backward_equals_separate_calls():
    """attn_bwd_group runs several one-pass blocks in one launch: dK and dV
    equal the per-block attn_bwd_ex(passes="fused") calls bit for bit, dQ (all
    blocks adding into one tiled accumulator) within fp32 rounding; causal and
    rectangular blocks, ragged lengths, a block without queries."""
    B, H, S = 1, 2, 1408
    scale = D ** -0.5
    g = torch.Generator(device="cuda").manual_seed(41)
    q, k, v, do = (torch.randn(B, S, H, D, generator=g, device="cuda").to(torch.bfloat16) for _ in range(4))
    lse = torch.randn(B, H, S, generator=g, device="cuda") + 6.0  # any statistics do for an equality check
    delta = torch.randn(B, H, S, generator=g, device="cuda")
    tasks = [(0, 384, 0, 384, 1),        # causal diagonal block
             (384, 300, 384, 513, 0),    # rectangular, ragged both ways
             (768, 640, 1000, 300, 0),   # ragged keys
             (128, 200, 897, 103, 0),    # overlapping query rows with another block (dQ adds)
             (0, 0, 1300, 100, 0)]       # no queries: its dK/dV rows are zeroed
    f32 = lambda: torch.full((B, S, H, D), 3.0, device="cuda")  # noqa: E731
    t1, dk1, dv1 = lcb.dq_tiles_zeros(B, H, S, "cuda"), f32(), f32()
    lcb.attn_bwd_group(q, k, v, lse, delta, do, t1, dk1, dv1, tasks, scale, accumulate=False)
    t2, dk2, dv2 = lcb.dq_tiles_zeros(B, H, S, "cuda"), f32(), f32()
    for qo, ql, ko, kl, causal in tasks:
        qs, ks = slice(qo, qo + ql), slice(ko, ko + kl)
        lcb.attn_bwd_ex(q[:, qs], k[:, ks], v[:, ks], lse[:, :, qs], delta[:, :, qs], do[:, qs],
                        t2[:, :, qo // 128:], dk2[:, ks], dv2[:, ks], bool(causal), scale, accumulate=False,
                        passes="fused")
    torch.cuda.synchronize()
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert (dk1[:, 1300:1400] == 0).all() and (dv1[:, 1300:1400] == 0).all()
    assert (dk1[:, 1400:] == 3.0).all()  # rows of no block are left alone
    assert torch.allclose(untile_f32(t1, S), untile_f32(t2, S), rtol=1e-5, atol=1e-5)
    assert torch.isfinite(untile_f32(t1, S)).all()


def test_batch_of_four_full_tensors():
    """B = 4, H = 8, S = 2048 (a batch of sequences), every element of O, LSE,
    dQ, dK and dV against the oracle. dV of the first keys sums many queries
    and reaches magnitudes where half a bf16 step exceeds 0.02, so the maximum
    bar is relative to max(1, |value|) here."""
    B, H, S = 4, 8, 2048
    q, k, v, do = gaussian_qkvdo(B, H, S, D, seed=44)
    o, lse = lcb.attn_fwd(q, k, v)
    dq, dk, dv = lcb.attn_bwd(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    ref = oracle.attn_bwd(to64(q), to64(k), to64(v), to64(do), True, D ** -0.5)
    assert_bf16_close(to64(o), ref["o"], "O B4")
    assert_lse_close(to64(lse), ref["lse"])
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_bf16_close_scaled(to64(got), ref[name], f"{name} B4")


@pytest.mark.parametrize("B,H,S", [(2, 3, 300), (1, 32, 4096), (1, 1, 1)])
def test_dq_untile_both_store_widths(B, H, S):
    """lcb_dq_untile is a layout change plus one bf16 rounding: bit-exact
    against undoing the documented tile layout in torch, through the 16-byte
    store path (aligned contiguous rows) and the 8-byte path (a row stride of
    H*128 + 4 elements); the padding of the strided rows is not touched."""
    g = torch.Generator(device="cuda").manual_seed(B * 1000 + H * 10 + S)
    tiles = torch.randn(B, H, (S + 127) // 128, 128 * 128, generator=g, device="cuda") * 3
    want = untile_f32(tiles, S).to(torch.bfloat16)
    dq = lcb.dq_untile(tiles, torch.empty(B, S, H, D, dtype=torch.bfloat16, device="cuda"))
    buf = torch.full((B, S, H * D + 4), 7.0, dtype=torch.bfloat16, device="cuda")
    dq_s = lcb.dq_untile(tiles, buf.as_strided((B, S, H, D), (S * (H * D + 4), H * D + 4, D, 1)))
    torch.cuda.synchronize()
    assert torch.equal(dq, want)
    assert torch.equal(dq_s, want)
    assert (buf[:, :, H * D:] == 7.0).all()
