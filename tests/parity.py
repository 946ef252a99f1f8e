"""Tolerances and comparison helpers shared by the GPU parity tests.

Bars (fixed before any kernel ran): bf16 outputs (O, dQ, dK, dV) within
max-abs 2e-2 and mean-abs 2e-3 of the fp64 oracle; LSE within 1e-3
absolute; schedule and index work bit-exact.
"""

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def to64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def err_stats(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    rel_l2 = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))
    return float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0, rel_l2


def assert_bf16_close(got, want, name, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    mx, mean, rel = err_stats(got, want)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    assert mx <= max_abs and mean <= mean_abs, (
        f"{name}: max-abs {mx:.3e} (bar {max_abs}), mean-abs {mean:.3e} (bar {mean_abs}), rel-L2 {rel:.3e}")
    return mx, mean, rel


def assert_lse_close(got, want, name="lse", tol=LSE_ABS):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    inf_g, inf_w = np.isneginf(got), np.isneginf(want)
    assert np.array_equal(inf_g, inf_w), f"{name}: -inf pattern differs"
    fin = ~inf_w
    if fin.any():
        mx = float(np.abs(got[fin] - want[fin]).max())
        assert mx <= tol, f"{name}: max-abs {mx:.3e} (bar {tol})"
        return mx
    return 0.0


def rows_budget(default):
    """Sampled rows per head for the large-size parity tests (LCB_PARITY_ROWS
    raises or lowers it)."""
    return int(os.environ.get("LCB_PARITY_ROWS", default))


def head64(t, h):
    """One head of a [B, S, H, D] device tensor as fp64 numpy [B, S, 1, D]."""
    return t[:, :, h:h + 1].float().cpu().numpy().astype(np.float64)


def map_heads(fn, heads, workers=None):
    """fn(h) for every head on a thread pool. numpy's BLAS calls and large
    ufunc loops release the GIL, so the per-head oracle calls overlap; the
    oracle itself is unchanged."""
    workers = workers or min(8, os.cpu_count() or 1)
    with ThreadPoolExecutor(max_workers=max(1, min(workers, len(heads)))) as ex:
        return list(ex.map(fn, heads))
