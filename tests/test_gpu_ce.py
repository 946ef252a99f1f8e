"""GPU parity of the cross-entropy loss head (in-place backward) against the
fp64 oracle: loss and LSE within 1e-3 absolute (the attention LSE bar); every
bf16 gradient element within one bf16 step of the exact value plus 2e-6 (the
fp32 arithmetic of softmax - onehot)."""

import numpy as np
import pytest
import torch

import oracle
import long_context_causal_blockwise_gb300 as lcb
from parity import to64

pytestmark = pytest.mark.gpu


def _case(N, V, seed, scale=3.0, ignore_frac=0.1):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = (torch.randn(N, V, generator=g, device="cuda") * scale).to(torch.bfloat16)
    y = torch.randint(0, V, (N,), generator=g, device="cuda")
    drop = torch.rand(N, generator=g, device="cuda") < ignore_frac
    y = torch.where(drop, torch.full_like(y, -100), y)
    return x, y


def _check(x0, y, loss, lse, grad, rows=None, dloss=None):
    rows = np.arange(x0.shape[0]) if rows is None else rows
    xr = to64(x0[rows])
    yr = y[rows].cpu().numpy()
    want_loss, want_lse = oracle.ce_fwd(xr, yr)
    assert np.abs(to64(lse[rows]) - want_lse).max() <= 1e-3
    if loss is not None:
        assert np.abs(to64(loss[rows]) - want_loss).max() <= 1e-3
    if grad is not None:
        g = 1.0 if dloss is None else to64(dloss[rows])
        want = oracle.ce_grad(xr, yr, g)
        # one bf16 step of the exact value (output rounding) plus the fp32 arithmetic of p and p - 1
        # (a given LSE, mode "bwd", enters x - LSE with its fp32 rounding: |LSE| 2^-23 more)
        slack = 2e-6 + (0.0 if dloss is None else 2.0 ** -23 * np.abs(to64(lse[rows]))[:, None])
        err = np.abs(to64(grad[rows]) - want) / (2.0 ** -7 * np.abs(want) + slack)
        assert err.max() <= 1.0, err.max()


@pytest.mark.parametrize("N,V", [(100, 1000), (37, 1001), (5, 8), (3, 1), (5000, 1000), (300, 50304), (400, 57344),
                                 (40, 128256), (9, 120001), (1, 128256)])
def test_ce_modes_vs_oracle(N, V):
    """fwd, fwd_bwd (in place) and bwd from a saved LSE. Rows are streamed
    through registers: 16-byte loads where a row's address and length are
    multiples of 16 bytes (V = 1000, 8, 50304, 57344, 128256), one logit at a
    time otherwise (V = 1001, 1, 120001); N = 5000 gives each persistent CTA
    many rows. The three launch shapes: five 256-thread CTAs per SM (V up to
    about 44000), four (V = 50304), one 1024-thread CTA per SM (V = 57344 and
    above)."""
    x, y = _case(N, V, seed=N + V)
    x0 = x.clone()
    loss, lse = lcb.cross_entropy(x, y, mode="fwd")
    torch.cuda.synchronize()
    assert torch.equal(x, x0)  # read only
    _check(x0, y, loss, lse, None)
    loss2, lse2 = lcb.cross_entropy(x, y, mode="fwd_bwd")
    torch.cuda.synchronize()
    assert torch.equal(lse2, lse) and torch.equal(loss2, loss)
    _check(x0, y, loss2, lse2, x)
    x3 = x0.clone()
    dl = torch.rand(N, device="cuda") * 2 - 0.5
    lcb.cross_entropy(x3, y, mode="bwd", lse=lse, dloss=dl)
    torch.cuda.synchronize()
    _check(x0, y, None, lse, x3, dloss=dl)
    ign = (y == -100).cpu().numpy()
    assert (to64(loss)[ign] == 0).all() and (to64(x)[ign] == 0).all()


def test_ce_strided_rows_and_extremes():
    """A row stride wider than V (a vocabulary slice of a padded buffer), -inf
    logits, a dominant logit, and a label outside the vocabulary (loss NaN)."""
    N, V, W = 6, 4096, 4104
    g = torch.Generator(device="cuda").manual_seed(9)
    buf = (torch.randn(N, W, generator=g, device="cuda") * 2).to(torch.bfloat16)
    x = buf[:, :V]
    x[1, :2048] = float("-inf")
    x[2, 17] = 90.0
    y = torch.tensor([5, 3000, 17, -100, 4095, 7], device="cuda")
    x0 = x.clone()
    pad0 = buf[:, V:].clone()
    loss, lse = lcb.cross_entropy(x, y, mode="fwd_bwd")
    torch.cuda.synchronize()
    _check(x0, y, loss, lse, x)
    assert torch.equal(buf[:, V:], pad0)  # the padding is not touched
    assert float(loss[2]) < 1e-6
    y_bad = torch.tensor([V + 3], device="cuda")
    loss_b, _ = lcb.cross_entropy(x0[:1].clone(), y_bad, mode="fwd")
    torch.cuda.synchronize()
    assert torch.isnan(loss_b).all()


def test_ce_llama_vocab_32768_tokens_sampled():
    """Llama-2 vocabulary (V = 32000) over a 32768-token sequence, fused
    fwd+bwd in place, checked on 2048 sampled rows plus the first and last."""
    N, V = 32768, 32000
    x, y = _case(N, V, seed=3)
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 2048, replace=False)]))
    rows_d = torch.as_tensor(rows, device="cuda")
    x_rows = x[rows_d].clone()
    loss, lse = lcb.cross_entropy(x, y, mode="fwd_bwd")
    torch.cuda.synchronize()
    _check(x_rows, y[rows_d], loss[rows_d], lse[rows_d], x[rows_d])
    assert torch.isfinite(x).all()


def test_ce_wide_vocabulary_all_rows():
    """V = 100000 (200 KB rows, the 1024-thread launch shape), fused forward
    and backward, every row checked."""
    N, V = 48, 100000
    x, y = _case(N, V, seed=17, ignore_frac=0.0)
    x0 = x.clone()
    loss, lse = lcb.cross_entropy(x, y, mode="fwd_bwd")
    torch.cuda.synchronize()
    _check(x0, y, loss, lse, x)
