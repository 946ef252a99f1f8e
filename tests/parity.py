"""Tolerances and comparison helpers shared by the GPU parity tests.

Bars (fixed before any kernel ran): bf16 outputs (O, dQ, dK, dV) within
max-abs 2e-2 and mean-abs 2e-3 of the fp64 oracle; LSE within 1e-3
absolute; schedule and index work bit-exact.
"""

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor, ThreadPoolExecutor

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


def assert_bf16_close_scaled(got, want, name, max_rel=MAX_ABS, mean_abs=MEAN_ABS):
    """The bf16 bars with the maximum taken relative to max(1, |want|): for
    outputs larger than 1 in magnitude half a bf16 step alone reaches the
    absolute bar (0.0156 at 4, 0.031 at 8), so there the bar is relative."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    scaled = np.abs(got - want) / np.maximum(1.0, np.abs(want))
    mx, mean, rel = err_stats(got, want)
    assert scaled.max() <= max_rel and mean <= mean_abs, (
        f"{name}: scaled max {scaled.max():.3e} (bar {max_rel}), max-abs {mx:.3e}, mean-abs {mean:.3e} "
        f"(bar {mean_abs}), rel-L2 {rel:.3e}")


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


def _bf16_bits_to_f64(a):
    """bf16 values stored as uint16 bit patterns -> fp64 (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rows_job(path, shape, h, rows, causal, scale):
    """Worker: oracle.attn_rows on head h of the bf16 q, k, v, dO held in a file."""
    import oracle
    arr = np.memmap(path, dtype=np.uint16, mode="r", shape=(4,) + tuple(shape))
    q, k, v, do = (_bf16_bits_to_f64(arr[i][:, :, h:h + 1, :]) for i in range(4))
    del arr
    return oracle.attn_rows(q, k, v, do, rows, causal, scale)


def _scratch_dir(nbytes):
    """/dev/shm when it has room for the inputs, else the temp directory."""
    import shutil
    import tempfile
    for d in ("/dev/shm", tempfile.gettempdir()):
        try:
            if os.path.isdir(d) and shutil.disk_usage(d).free > 2 * nbytes:
                return d
        except OSError:
            pass
    return tempfile.gettempdir()


def oracle_rows_by_head(q, k, v, do, rows, causal, scale, workers=None):
    """oracle.attn_rows for every head of device tensors q, k, v, dO [B, S, H, D]
    (bf16), one head per task on a pool of spawned processes with one BLAS
    thread each; the inputs reach the workers through a scratch file (bf16
    bit patterns). Returns the per-head result dicts in head order."""
    import tempfile
    import torch
    B, S, H, D = q.shape
    nbytes = 4 * q.numel() * 2
    fd, path = tempfile.mkstemp(prefix="lcb_oracle_", suffix=".bin", dir=_scratch_dir(nbytes))
    os.close(fd)
    try:
        mm = np.memmap(path, dtype=np.uint16, mode="w+", shape=(4, B, S, H, D))
        host = torch.from_numpy(mm.view(np.int16))
        for i, t in enumerate((q, k, v, do)):
            host[i].copy_(t.contiguous().view(torch.int16))
        del host
        mm.flush()
        del mm
        workers = workers or min(16, os.cpu_count() or 1, H)
        saved = {n: os.environ.get(n) for n in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
        os.environ.update({n: "1" for n in saved})  # inherited by the spawned workers
        try:
            with ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
                futs = [ex.submit(_rows_job, path, (B, S, H, D), h, rows, causal, scale) for h in range(H)]
                return [f.result() for f in futs]
        finally:
            for n, val in saved.items():
                if val is None:
                    os.environ.pop(n, None)
                else:
                    os.environ[n] = val
    finally:
        os.unlink(path)
