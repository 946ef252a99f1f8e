"""fp64 CPU oracle for exact softmax attention, forward and backward.

TEST INFRASTRUCTURE (see the package header): only tests/, the smoke check and
the bench's CPU-baseline leg may call this module.

Definition followed (the textbook attention that Flash Attention reaches
exactly, "EasyContext核心技术解析：序列并行与Flash Attention的完美结合",
§2 "Flash Attention优化"; full attention, "EasyContext：用最少资源扩展大模型至
百万Token"). For each batch b, head h and query row i:

    s_ij   = scale * q_i . k_j           for visible j
    LSE_i  = ln sum_j exp(s_ij)           (natural log, scale included)
    P_ij   = exp(s_ij - LSE_i)
    O_i    = sum_j P_ij v_j

Visible means j <= i when causal (square case, Sq == Sk), every j < Sk
otherwise. A row with no visible key has LSE = -inf, O = 0 and zero gradients.

Backward for an upstream gradient dO of O:

    Delta_i = dO_i . O_i
    dP_ij   = dO_i . v_j
    dS_ij   = P_ij (dP_ij - Delta_i)
    dQ_i    = scale * sum_j dS_ij k_j
    dK_j    = scale * sum_i dS_ij q_i
    dV_j    = sum_i P_ij dO_i

Layouts: q, k, v, dO, O, dQ, dK, dV are [B, S, H, D]; LSE and Delta are
[B, H, S]. Inputs of any float dtype are upcast to fp64 before any arithmetic.
The full softmax rows are materialised (in row panels, to bound memory); the
only stabilisation is subtracting the row maximum before exp.
"""

import numpy as np

# Rows per panel are chosen so that a panel of scores holds about 2**25 fp64
# values (256 MB); small problems take a single panel.
_PANEL_ELEMS = 1 << 25


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _panel_rows(n_keys):
    return max(1, min(1 << 16, _PANEL_ELEMS // max(1, n_keys)))


def _visible(rows, n_keys, causal):
    """Boolean [len(rows), n_keys]: key j is visible to query row i."""
    j = np.arange(n_keys)
    if causal:
        return j[None, :] <= np.asarray(rows)[:, None]
    return np.ones((len(rows), n_keys), dtype=bool)


def _softmax_rows(s, vis):
    """Softmax of scaled scores s over the visible keys.

    Returns (P, LSE). P is zero on hidden keys; a row with no visible key
    gets P = 0 and LSE = -inf.
    """
    s = np.where(vis, s, -np.inf)
    if s.shape[1] == 0:
        return np.zeros_like(s), np.full(s.shape[0], -np.inf)
    m = s.max(axis=1)
    m0 = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m0[:, None])
    z = e.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(z > 0, m0 + np.log(np.where(z > 0, z, 1.0)), -np.inf)
        p = np.where(z[:, None] > 0, e / np.where(z > 0, z, 1.0)[:, None], 0.0)
    return p, lse


def _check(q, k, v, causal):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, S, H, D]")
    B, Sq, H, D = q.shape
    if k.shape[0] != B or k.shape[2] != H or k.shape[3] != D or v.shape != k.shape:
        raise ValueError("k and v must be [B, Sk, H, D] matching q")
    if causal and Sq != k.shape[1]:
        raise ValueError("causal attention is defined here for Sq == Sk only")
    return B, Sq, k.shape[1], H, D


def attn_probs(q, k, v, causal, scale):
    """The full probability matrix P [B, H, Sq, Sk] (small problems only)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Sk, H, D = _check(q, k, v, causal)
    P = np.zeros((B, H, Sq, Sk))
    rows = np.arange(Sq)
    vis = _visible(rows, Sk, causal)
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, :, h, :] @ k[b, :, h, :].T)
            P[b, h], _ = _softmax_rows(s, vis)
    return P


def attn_fwd(q, k, v, causal, scale):
    """Forward: returns (O [B,Sq,H,D] fp64, LSE [B,H,Sq] fp64)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, Sk, H, D = _check(q, k, v, causal)
    O = np.zeros((B, Sq, H, D))
    LSE = np.full((B, H, Sq), -np.inf)
    step = _panel_rows(Sk)
    for b in range(B):
        for h in range(H):
            kh, vh = k[b, :, h, :], v[b, :, h, :]
            for r0 in range(0, Sq, step):
                rows = np.arange(r0, min(Sq, r0 + step))
                s = scale * (q[b, rows, h, :] @ kh.T)
                p, lse = _softmax_rows(s, _visible(rows, Sk, causal))
                O[b, rows, h, :] = p @ vh
                LSE[b, h, rows] = lse
    return O, LSE


def attn_bwd(q, k, v, do, causal, scale):
    """Forward and backward by the definition.

    Returns a dict with o, lse, delta, dq, dk, dv (fp64, layouts as above).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Sq, Sk, H, D = _check(q, k, v, causal)
    out = {
        "o": np.zeros((B, Sq, H, D)),
        "lse": np.full((B, H, Sq), -np.inf),
        "delta": np.zeros((B, H, Sq)),
        "dq": np.zeros((B, Sq, H, D)),
        "dk": np.zeros((B, Sk, H, D)),
        "dv": np.zeros((B, Sk, H, D)),
    }
    step = _panel_rows(Sk)
    for b in range(B):
        for h in range(H):
            kh, vh = k[b, :, h, :], v[b, :, h, :]
            for r0 in range(0, Sq, step):
                rows = np.arange(r0, min(Sq, r0 + step))
                qh, doh = q[b, rows, h, :], do[b, rows, h, :]
                p, lse = _softmax_rows(scale * (qh @ kh.T), _visible(rows, Sk, causal))
                o = p @ vh
                delta = np.sum(doh * o, axis=1)
                dp = doh @ vh.T
                ds = p * (dp - delta[:, None])
                out["o"][b, rows, h, :] = o
                out["lse"][b, h, rows] = lse
                out["delta"][b, h, rows] = delta
                out["dq"][b, rows, h, :] = scale * (ds @ kh)
                out["dk"][b, :, h, :] += scale * (ds.T @ qh)
                out["dv"][b, :, h, :] += p.T @ doh
    return out


def attn_bwd_given_stats(q, k, v, do, lse, delta, causal, scale):
    """Backward of one block of keys with the row statistics given from outside.

    P_ij = exp(s_ij - LSE_i) and dS_ij = P_ij (dP_ij - Delta_i), with LSE and
    Delta supplied by the caller ([B, H, Sq]). When LSE and Delta are the
    statistics of attention over ALL keys, summing this over disjoint key
    blocks gives the monolithic gradients: this is how the steps of a ring
    backward compose (ring attention, "EasyContext核心技术解析…" §1
    "序列并行技术"). Returns (dq [B,Sq,H,D], dk [B,Sk,H,D], dv [B,Sk,H,D]).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    lse, delta = _f64(lse), _f64(delta)
    B, Sq, Sk, H, D = _check(q, k, v, causal)
    dq = np.zeros((B, Sq, H, D))
    dk = np.zeros((B, Sk, H, D))
    dv = np.zeros((B, Sk, H, D))
    step = _panel_rows(Sk)
    for b in range(B):
        for h in range(H):
            kh, vh = k[b, :, h, :], v[b, :, h, :]
            for r0 in range(0, Sq, step):
                rows = np.arange(r0, min(Sq, r0 + step))
                qh, doh = q[b, rows, h, :], do[b, rows, h, :]
                vis = _visible(rows, Sk, causal)
                s = np.where(vis, scale * (qh @ kh.T), -np.inf)
                l_r = lse[b, h, rows]
                l0 = np.where(np.isfinite(l_r), l_r, 0.0)
                p = np.where(vis & np.isfinite(l_r)[:, None], np.exp(s - l0[:, None]), 0.0)
                ds = p * (doh @ vh.T - delta[b, h, rows][:, None])
                dq[b, rows, h, :] = scale * (ds @ kh)
                dk[b, :, h, :] += scale * (ds.T @ qh)
                dv[b, :, h, :] += p.T @ doh
    return dq, dk, dv


def attn_rows(q, k, v, do, rows, causal, scale):
    """Row-local outputs for a sample of query rows, every batch and head.

    O_i, LSE_i, Delta_i and dQ_i depend only on query row i, so a sample of
    rows is checked exactly without the rest. When causal, a panel of rows
    only forms the keys up to its last row: the keys after a row are not
    visible to it, contribute exactly zero, and are left out.
    Returns a dict with o [B,R,H,D], lse [B,H,R], delta [B,H,R] and (when do
    is given) dq [B,R,H,D].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    do = None if do is None else _f64(do)
    B, Sq, Sk, H, D = _check(q, k, v, causal)
    rows = np.asarray(rows, dtype=np.int64)
    R = len(rows)
    out = {
        "o": np.zeros((B, R, H, D)),
        "lse": np.full((B, H, R), -np.inf),
        "delta": np.zeros((B, H, R)),
        "dq": None if do is None else np.zeros((B, R, H, D)),
    }
    step = _panel_rows(Sk)
    for b in range(B):
        for h in range(H):
            for a0 in range(0, R, step):
                sel = np.arange(a0, min(R, a0 + step))
                rr = rows[sel]
                nk = min(Sk, int(rr.max()) + 1) if causal else Sk  # keys any row of the panel can see
                kh, vh = k[b, :nk, h, :], v[b, :nk, h, :]
                p, lse = _softmax_rows(scale * (q[b, rr, h, :] @ kh.T), _visible(rr, nk, causal))
                o = p @ vh
                out["o"][b, sel, h, :] = o
                out["lse"][b, h, sel] = lse
                if do is not None:
                    doh = do[b, rr, h, :]
                    delta = np.sum(doh * o, axis=1)
                    ds = p * (doh @ vh.T - delta[:, None])
                    out["delta"][b, h, sel] = delta
                    out["dq"][b, sel, h, :] = scale * (ds @ kh)
    return out


def attn_key_rows(q, k, v, do, keys, heads, causal, scale):
    """dK and dV for a sample of key rows on a subset of heads, every batch.

    dK_j and dV_j sum over all query rows i, and each term needs LSE_i and
    Delta_i, i.e. the whole softmax row i. Every query row that can see a
    sampled key is therefore formed in full (in panels); only the sampled key
    columns are reduced. When causal, query rows i < min(keys) see none of the
    sampled keys (P_ij = 0 for j > i) and are skipped, so keys sampled near the
    end of a long sequence are cheap.
    Returns (dk [B,K,len(heads),D], dv [B,K,len(heads),D]).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Sq, Sk, H, D = _check(q, k, v, causal)
    keys = np.asarray(keys, dtype=np.int64)
    dk = np.zeros((B, len(keys), len(heads), D))
    dv = np.zeros((B, len(keys), len(heads), D))
    step = _panel_rows(Sk)
    first = int(keys.min()) if (causal and len(keys)) else 0
    for b in range(B):
        for hi, h in enumerate(heads):
            kh, vh = k[b, :, h, :], v[b, :, h, :]
            for r0 in range(first, Sq, step):
                rows = np.arange(r0, min(Sq, r0 + step))
                qh, doh = q[b, rows, h, :], do[b, rows, h, :]
                p, _ = _softmax_rows(scale * (qh @ kh.T), _visible(rows, Sk, causal))
                delta = np.sum(doh * (p @ vh), axis=1)
                pk = p[:, keys]
                dsk = pk * (doh @ vh[keys].T - delta[:, None])
                dk[b, :, hi, :] += scale * (dsk.T @ qh)
                dv[b, :, hi, :] += pk.T @ doh
    return dk, dv
