"""Parity at the long-context sizes, on outputs the oracle can form one by one.

  * Llama-2-13B attention layer: B=1, H=40, D=128, S=262144, causal.
  * Long-context stress: B=1, H=32, D=128, S=524288, causal, Q and K
    pre-rotated by RoPE with theta = 1e6 over positions 0..S-1.

Checked against the fp64 oracle: O, LSE and dQ on 4096 sampled query rows of
every head (row-local; LCB_PARITY_ROWS changes the count); dK and dV on the
last keys of the sequence for two heads (under the causal mask only the final
queries see them, so the oracle forms just those rows in full); and the sum
rules sum_j dV_j = sum_i dO_i and sum_j dK_j = 0 on every head, which hold at
any size.
"""

import numpy as np
import pytest
import torch

import oracle
import long_context_causal_blockwise_gb300 as lcb
from long_context_causal_blockwise_gb300.inputs import gaussian_qkvdo, sample_rows
from parity import assert_bf16_close, assert_lse_close, head64, map_heads, oracle_rows_by_head, rows_budget, to64

pytestmark = pytest.mark.gpu
D = 128


def _check_large(H, S, rope_theta, seed, n_rows, tail):
    scale = D ** -0.5
    q, k, v, do = gaussian_qkvdo(1, H, S, D, seed=seed, rope_theta=rope_theta)
    o, lse = lcb.attn_fwd(q, k, v)
    dq, dk, dv = lcb.attn_bwd(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    for t, name in ((o, "O"), (dq, "dQ"), (dk, "dK"), (dv, "dV")):
        assert torch.isfinite(t).all(), f"{name}: non-finite values"
    rows = sample_rows(S, n_rows, seed=seed + 11)
    rows_d = torch.as_tensor(rows, device="cuda")
    keys = np.arange(S - tail, S)
    keys_d = torch.as_tensor(keys, device="cuda")

    refs = oracle_rows_by_head(q, k, v, do, rows, True, scale)
    ends = (0, H - 1)
    krefs = map_heads(lambda h: oracle.attn_key_rows(*(head64(t, h) for t in (q, k, v, do)), keys, [0], True, scale),
                      list(ends))
    for h, (rdk, rdv) in zip(ends, krefs):
        assert_bf16_close(to64(dk[:, keys_d, h:h + 1]), rdk, f"dK tail keys S{S} head {h}")
        assert_bf16_close(to64(dv[:, keys_d, h:h + 1]), rdv, f"dV tail keys S{S} head {h}")
    assert_bf16_close(to64(o[:, rows_d]), np.concatenate([r["o"] for r in refs], 2), f"O sampled S{S}")
    assert_lse_close(to64(lse[:, :, rows_d]), np.concatenate([r["lse"] for r in refs], 1))
    assert_bf16_close(to64(dq[:, rows_d]), np.concatenate([r["dq"] for r in refs], 2), f"dQ sampled S{S}")
    sdv, sdo, sdk = dv.float().sum(1), do.float().sum(1), dk.float().sum(1)
    assert ((sdv - sdo).norm(dim=-1) <= 1e-2 * sdo.norm(dim=-1)).all()
    assert (sdk.norm(dim=-1) <= 1e-2 * dk.float().norm(dim=(1, 3))).all()


def test_config4_llama13b_layer_262144():
    _check_large(H=40, S=262144, rope_theta=None, seed=4, n_rows=rows_budget(4096), tail=96)


def test_config5_stress_524288_rope():
    _check_large(H=32, S=524288, rope_theta=1e6, seed=5, n_rows=rows_budget(4096), tail=64)
