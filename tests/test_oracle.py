"""Pins for the fp64 oracle, on the CPU.

Nothing here compares the oracle with itself: each test checks it against
something it does not compute (pure-Python brute force, closed forms, a
hand-derived worked example, invariants that hold for any input, central
finite differences), and the planted-mistake tests at the end show that a
plausible slip in the oracle's arithmetic fails at least one of these pins.
"""

import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as oatt

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


# ---------------------------------------------------------------- brute force

def _brute_fwd(q, k, v, causal, scale):
    """Pure-Python scalar attention: direct sums of math.exp, no max shift."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    O = [[[[0.0] * D for _ in range(H)] for _ in range(Sq)] for _ in range(B)]
    L = [[[0.0] * Sq for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                js = [j for j in range(Sk) if (not causal or j <= i)]
                w = []
                for j in js:
                    dot = 0.0
                    for d in range(D):
                        dot += float(q[b, i, h, d]) * float(k[b, j, h, d])
                    w.append(math.exp(scale * dot))
                z = sum(w)
                L[b][h][i] = math.log(z)
                for d in range(D):
                    O[b][i][h][d] = sum(w[t] * float(v[b, j, h, d]) for t, j in enumerate(js)) / z
    return np.array(O), np.array(L)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,H,S,D", [(1, 1, 1, 4), (2, 2, 7, 8), (1, 2, 16, 3)])
def test_forward_matches_scalar_brute_force(causal, B, H, S, D):
    rng = np.random.default_rng(1000 + S * 10 + D + int(causal))
    q, k, v = (_rand(rng, B, S, H, D) for _ in range(3))
    scale = 1.0 / math.sqrt(D)
    O, L = oracle.attn_fwd(q, k, v, causal, scale)
    Ob, Lb = _brute_fwd(q, k, v, causal, scale)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)


def test_forward_rectangular_noncausal_brute_force():
    rng = np.random.default_rng(7)
    q = _rand(rng, 1, 5, 2, 4)
    k, v = _rand(rng, 1, 11, 2, 4), _rand(rng, 1, 11, 2, 4)
    O, L = oracle.attn_fwd(q, k, v, False, 0.3)
    Ob, Lb = _brute_fwd(q, k, v, False, 0.3)
    np.testing.assert_allclose(O, Ob, atol=1e-12)
    np.testing.assert_allclose(L, Lb, atol=1e-12)


# ---------------------------------------------------------------- invariants of P

@pytest.mark.parametrize("causal", [True, False])
def test_probability_rows_sum_to_one_and_causal_zeros(causal):
    rng = np.random.default_rng(3)
    q, k, v = (_rand(rng, 1, 33, 2, 8) for _ in range(3))
    P = oracle.attn_probs(q, k, v, causal, 0.35)
    np.testing.assert_allclose(P.sum(axis=-1), 1.0, atol=1e-12)
    assert (P >= 0).all()
    if causal:
        iu = np.triu_indices(33, k=1)
        assert (P[:, :, iu[0], iu[1]] == 0.0).all()
        assert (P[:, :, np.arange(33), np.arange(33)] > 0).all()
    else:
        assert (P > 0).all()


# ---------------------------------------------------------------- closed forms

def test_single_key_row_is_exact():
    """S = 1, and row 0 of a causal problem: weight exactly 1 on key 0."""
    rng = np.random.default_rng(11)
    q, k, v = (_rand(rng, 2, 9, 3, 8) for _ in range(3))
    scale = 0.125
    O, L = oracle.attn_fwd(q, k, v, True, scale)
    assert np.array_equal(O[:, 0], v[:, 0])
    np.testing.assert_allclose(L[:, :, 0], scale * np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0]), atol=1e-13)
    O1, L1 = oracle.attn_fwd(q[:, :1], k[:, :1], v[:, :1], False, scale)
    assert np.array_equal(O1[:, 0], v[:, 0])


def test_zero_keys_give_prefix_mean():
    rng = np.random.default_rng(12)
    S = 40
    q, v = _rand(rng, 1, S, 2, 6), _rand(rng, 1, S, 2, 6)
    k = np.zeros_like(q)
    O, L = oracle.attn_fwd(q, k, v, True, 0.4)
    prefix_mean = np.cumsum(v, axis=1) / np.arange(1, S + 1)[None, :, None, None]
    np.testing.assert_allclose(O, prefix_mean, atol=1e-12)
    np.testing.assert_allclose(L, np.log(np.arange(1, S + 1))[None, None, :].repeat(2, 1), atol=1e-12)
    On, Ln = oracle.attn_fwd(q, k, v, False, 0.4)
    np.testing.assert_allclose(On, np.broadcast_to(v.mean(axis=1, keepdims=True), v.shape), atol=1e-12)
    np.testing.assert_allclose(Ln, math.log(S), atol=1e-12)


def test_constant_values_give_constant_output():
    rng = np.random.default_rng(13)
    q, k = _rand(rng, 1, 25, 2, 8, scale=3.0), _rand(rng, 1, 25, 2, 8, scale=3.0)
    v = np.ones_like(q)
    for causal in (True, False):
        O, _ = oracle.attn_fwd(q, k, v, causal, 0.5)
        np.testing.assert_allclose(O, 1.0, atol=1e-12)


def test_peaked_scores_pick_the_argmax_value():
    """Scores around 1e3 with a lead of > 40: the max shift must keep this finite."""
    S, D = 12, 4
    rng = np.random.default_rng(14)
    v = _rand(rng, 1, S, 1, D)
    # k_j = (j, 0, 0, 0) and q_i = (1000, 0, 0, 0): the latest visible key wins by 1000.
    k = np.zeros((1, S, 1, D))
    k[0, :, 0, 0] = np.arange(S)
    q = np.zeros((1, S, 1, D))
    q[0, :, 0, 0] = 1000.0
    O, L = oracle.attn_fwd(q, k, v, True, 1.0)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    np.testing.assert_allclose(O[0, :, 0], v[0, :, 0], atol=1e-12)
    np.testing.assert_allclose(L[0, 0], 1000.0 * np.arange(S), rtol=1e-15, atol=1e-9)
    On, _ = oracle.attn_fwd(q, k, v, False, 1.0)
    np.testing.assert_allclose(On[0, :, 0], np.broadcast_to(v[0, -1, 0], (S, D)), atol=1e-12)


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *toks = line.split()
            vals.setdefault(key, []).append(toks)
    return vals


def _num(tok):
    return float(eval(tok, {"__builtins__": {}}, {"ln": math.log}))


def test_worked_example_golden():
    g = _read_golden("worked_causal_s3_d2.txt")
    arr = {k: np.array([_num(t) for t in v[0]]) for k, v in g.items()}
    q = arr["q"].reshape(1, 3, 1, 2)
    k = arr["k"].reshape(1, 3, 1, 2)
    v = arr["v"].reshape(1, 3, 1, 2)
    do = arr["do"].reshape(1, 3, 1, 2)
    r = oracle.attn_bwd(q, k, v, do, True, 1.0)
    np.testing.assert_allclose(r["o"].ravel(), arr["o"], atol=1e-14)
    np.testing.assert_allclose(r["lse"].ravel(), arr["lse"], atol=1e-14)
    np.testing.assert_allclose(r["delta"].ravel(), arr["delta"], atol=1e-14)
    np.testing.assert_allclose(r["dq"].ravel(), arr["dq"], atol=1e-14)
    np.testing.assert_allclose(r["dk"].ravel(), arr["dk"], atol=1e-14)
    np.testing.assert_allclose(r["dv"].ravel(), arr["dv"], atol=1e-14)


# ---------------------------------------------------------------- backward

def _loss(q, k, v, do, causal, scale):
    O, _ = oracle.attn_fwd(q, k, v, causal, scale)
    return float(np.sum(do * O))


@pytest.mark.parametrize("causal", [True, False])
def test_backward_central_finite_differences(causal):
    rng = np.random.default_rng(21 + int(causal))
    B, S, H, D = 1, 8, 2, 4
    q, k, v, do = (_rand(rng, B, S, H, D) for _ in range(4))
    scale = 0.7
    r = oracle.attn_bwd(q, k, v, do, causal, scale)
    h = 1e-5
    for name, x, g in (("q", q, r["dq"]), ("k", k, r["dk"]), ("v", v, r["dv"])):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], do, causal, scale)
                        - _loss(args_m["q"], args_m["k"], args_m["v"], do, causal, scale)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-7, err_msg=name)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_sum_invariants(causal):
    """sum_j P_ij = 1 gives sum_j dV_j = sum_i dO_i; sum_j dS_ij = 0 gives sum_j dK_j = 0."""
    rng = np.random.default_rng(31)
    q, k, v, do = (_rand(rng, 2, 37, 3, 16) for _ in range(4))
    r = oracle.attn_bwd(q, k, v, do, causal, 0.25)
    np.testing.assert_allclose(r["dv"].sum(axis=1), do.sum(axis=1), atol=1e-11)
    np.testing.assert_allclose(r["dk"].sum(axis=1), 0.0, atol=1e-11)
    # and Delta is dO . O row by row
    np.testing.assert_allclose(r["delta"], np.einsum("bshd,bshd->bhs", do, r["o"]), atol=1e-12)


def test_given_stats_block_sum_equals_monolithic():
    """With global LSE and Delta, block gradients over a key split add up."""
    rng = np.random.default_rng(41)
    q, k, v, do = (_rand(rng, 1, 20, 2, 8) for _ in range(4))
    full = oracle.attn_bwd(q, k, v, do, False, 0.3)
    dq = np.zeros_like(q)
    dk_parts, dv_parts = [], []
    for a, b in ((0, 7), (7, 13), (13, 20)):
        gq, gk, gv = oracle.attn_bwd_given_stats(q, k[:, a:b], v[:, a:b], do, full["lse"], full["delta"], False, 0.3)
        dq += gq
        dk_parts.append(gk)
        dv_parts.append(gv)
    np.testing.assert_allclose(dq, full["dq"], atol=1e-12)
    np.testing.assert_allclose(np.concatenate(dk_parts, axis=1), full["dk"], atol=1e-12)
    np.testing.assert_allclose(np.concatenate(dv_parts, axis=1), full["dv"], atol=1e-12)


def test_sampled_rows_agree_with_full():
    rng = np.random.default_rng(51)
    q, k, v, do = (_rand(rng, 2, 50, 2, 8) for _ in range(4))
    full = oracle.attn_bwd(q, k, v, do, True, 0.3)
    rows = np.array([0, 1, 17, 48, 49])
    rr = oracle.attn_rows(q, k, v, do, rows, True, 0.3)
    np.testing.assert_allclose(rr["o"], full["o"][:, rows], atol=1e-13)
    np.testing.assert_allclose(rr["lse"], full["lse"][:, :, rows], atol=1e-13)
    np.testing.assert_allclose(rr["dq"], full["dq"][:, rows], atol=1e-13)
    np.testing.assert_allclose(rr["delta"], full["delta"][:, :, rows], atol=1e-13)
    # unsorted rows (each panel forms only the keys its rows can see) and a non-causal sample
    rows2 = np.array([33, 2, 49, 10])
    rr2 = oracle.attn_rows(q, k, v, do, rows2, True, 0.3)
    np.testing.assert_allclose(rr2["o"], full["o"][:, rows2], atol=1e-13)
    np.testing.assert_allclose(rr2["dq"], full["dq"][:, rows2], atol=1e-13)
    nc = oracle.attn_bwd(q, k, v, do, False, 0.3)
    rr3 = oracle.attn_rows(q, k, v, do, rows2, False, 0.3)
    np.testing.assert_allclose(rr3["o"], nc["o"][:, rows2], atol=1e-13)
    np.testing.assert_allclose(rr3["dq"], nc["dq"][:, rows2], atol=1e-13)
    keys = np.array([0, 5, 49])
    dk, dv = oracle.attn_key_rows(q, k, v, do, keys, [1], True, 0.3)
    np.testing.assert_allclose(dk[:, :, 0], full["dk"][:, keys, 1], atol=1e-12)
    np.testing.assert_allclose(dv[:, :, 0], full["dv"][:, keys, 1], atol=1e-12)
    # tail keys: only query rows at or after the first sampled key are formed
    tail = np.array([40, 44, 49])
    dk, dv = oracle.attn_key_rows(q, k, v, do, tail, [0, 1], True, 0.3)
    np.testing.assert_allclose(dk, full["dk"][:, tail], atol=1e-12)
    np.testing.assert_allclose(dv, full["dv"][:, tail], atol=1e-12)


def test_empty_rows():
    q = np.ones((1, 3, 1, 2))
    k = np.ones((1, 0, 1, 2))
    O, L = oracle.attn_fwd(q, k, k, False, 1.0)
    assert (O == 0).all() and np.isneginf(L).all()


# ---------------------------------------------------------------- merge

def test_merge_of_key_split_equals_monolithic():
    rng = np.random.default_rng(61)
    q = _rand(rng, 2, 9, 3, 8)
    k, v = _rand(rng, 2, 30, 3, 8), _rand(rng, 2, 30, 3, 8)
    O, L = oracle.attn_fwd(q, k, v, False, 0.4)
    Oa, La = oracle.attn_fwd(q, k[:, :11], v[:, :11], False, 0.4)
    Ob, Lb = oracle.attn_fwd(q, k[:, 11:], v[:, 11:], False, 0.4)
    Om, Lm = oracle.lse_merge(Oa, La, Ob, Lb)
    np.testing.assert_allclose(Om, O, atol=1e-12)
    np.testing.assert_allclose(Lm, L, atol=1e-12)
    # commutative, and associative over a three-way split
    Om2, Lm2 = oracle.lse_merge(Ob, Lb, Oa, La)
    np.testing.assert_allclose(Om2, Om, atol=1e-13)
    parts = [oracle.attn_fwd(q, k[:, a:b], v[:, a:b], False, 0.4) for a, b in ((0, 4), (4, 20), (20, 30))]
    left = oracle.lse_merge(*oracle.lse_merge(*parts[0], *parts[1]), *parts[2])
    right = oracle.lse_merge(*parts[0], *oracle.lse_merge(*parts[1], *parts[2]))
    np.testing.assert_allclose(left[0], O, atol=1e-12)
    np.testing.assert_allclose(right[0], O, atol=1e-12)
    np.testing.assert_allclose(left[1], right[1], atol=1e-13)


def test_merge_with_empty_sides():
    rng = np.random.default_rng(62)
    o = _rand(rng, 1, 4, 1, 3)
    lse = np.array([[[0.5, -np.inf, 2.0, -np.inf]]])
    empty_o = np.zeros_like(o)
    empty_l = np.full_like(lse, -np.inf)
    Om, Lm = oracle.lse_merge(o, lse, empty_o, empty_l)
    fin = np.isfinite(lse[0, 0])
    np.testing.assert_array_equal(Lm, lse)
    np.testing.assert_allclose(Om[0, fin], o[0, fin], atol=0)
    assert (Om[0, ~fin] == 0).all()
    Om, Lm = oracle.lse_merge(empty_o, empty_l, empty_o, empty_l)
    assert np.isneginf(Lm).all() and (Om == 0).all()
    # equal LSE on both sides: plain average and LSE + ln 2
    Om, Lm = oracle.lse_merge(o, np.zeros((1, 1, 4)), 3 * o, np.zeros((1, 1, 4)))
    np.testing.assert_allclose(Om, 2 * o, atol=1e-15)
    np.testing.assert_allclose(Lm, math.log(2.0), atol=1e-15)


# ---------------------------------------------------------------- zigzag

def test_zigzag_golden_s8_p2():
    g = _read_golden("zigzag_s8_p2.txt")
    perm, tasks = oracle.zigzag_schedule(8, 2)
    assert perm.tolist() == [int(t) for t in g["perm"][0]]
    got = [[t["rank"], t["step"], t["src"], t["kind"], t["q_off"], t["q_len"], t["k_off"], t["k_len"], t["causal"]]
           for t in tasks]
    assert got == [[int(x) for x in row] for row in g["task"]]


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("c", [1, 2, 5, 16])
def test_zigzag_covers_every_causal_pair_once(P, c):
    S = 2 * P * c
    if S > 256:
        pytest.skip("brute force kept to S <= 256")
    perm, tasks = oracle.zigzag_schedule(S, P)
    assert sorted(perm.tolist()) == list(range(S))
    count = oracle.zigzag_tasks_pairs(S, perm, tasks)
    want = np.tril(np.ones((S, S), dtype=np.int64))
    assert np.array_equal(count, want)
    # every rank does the same number of pairs: c^2 + c(c+1) + 2(P-1)c^2
    per_rank = {}
    for t in tasks:
        n = t["q_len"] * (t["q_len"] + 1) // 2 if t["causal"] else t["q_len"] * t["k_len"]
        per_rank[t["rank"]] = per_rank.get(t["rank"], 0) + n
    assert set(per_rank.values()) == {c * c + c * (c + 1) + 2 * (P - 1) * c * c}
    assert sum(per_rank.values()) == S * (S + 1) // 2


def test_zigzag_rejects_bad_sizes():
    for S, P in ((10, 3), (0, 1), (8, 0), (3, 2)):
        with pytest.raises(ValueError):
            oracle.zigzag_schedule(S, P)


@pytest.mark.parametrize("P", [1, 2, 4])
def test_zigzag_ring_emulation_equals_monolithic(P):
    """fp64: ring steps merged by LSE equal monolithic causal attention, and
    ring backward with the final merged statistics equals monolithic gradients."""
    S, H, D = 48, 2, 8
    rng = np.random.default_rng(70 + P)
    q, k, v, do = (_rand(rng, 1, S, H, D) for _ in range(4))
    scale = 0.35
    perm, tasks = oracle.zigzag_schedule(S, P)
    qz, kz, vz, doz = q[:, perm], k[:, perm], v[:, perm], do[:, perm]
    c2 = S // P
    Oz = np.zeros_like(qz)
    Lz = np.full((1, H, S), -np.inf)
    for t in tasks:
        qs = slice(t["q_off"], t["q_off"] + t["q_len"])
        ks = slice(t["k_off"], t["k_off"] + t["k_len"])
        Ob, Lb = oracle.attn_fwd(qz[:, qs], kz[:, ks], vz[:, ks], bool(t["causal"]), scale)
        Om, Lm = oracle.lse_merge(Oz[:, qs], Lz[:, :, qs], Ob, Lb)
        Oz[:, qs], Lz[:, :, qs] = Om, Lm
    full = oracle.attn_bwd(q, k, v, do, True, scale)
    inv = np.argsort(perm)
    np.testing.assert_allclose(Oz[:, inv], full["o"], atol=1e-12)
    np.testing.assert_allclose(Lz[:, :, inv], full["lse"], atol=1e-12)
    delta = np.einsum("bshd,bshd->bhs", doz, Oz)
    dq, dk, dv = np.zeros_like(qz), np.zeros_like(kz), np.zeros_like(vz)
    for t in tasks:
        qs = slice(t["q_off"], t["q_off"] + t["q_len"])
        ks = slice(t["k_off"], t["k_off"] + t["k_len"])
        gq, gk, gv = oracle.attn_bwd_given_stats(qz[:, qs], kz[:, ks], vz[:, ks], doz[:, qs],
                                                 Lz[:, :, qs], delta[:, :, qs], bool(t["causal"]), scale)
        dq[:, qs] += gq
        dk[:, ks] += gk
        dv[:, ks] += gv
    np.testing.assert_allclose(dq[:, inv], full["dq"], atol=1e-12)
    np.testing.assert_allclose(dk[:, inv], full["dk"], atol=1e-12)
    np.testing.assert_allclose(dv[:, inv], full["dv"], atol=1e-12)
    assert c2 * P == S


# ---------------------------------------------------------------- planted mistakes

def _pins_pass():
    """A compact run of independent pins; returns False if any of them fails."""
    checks = [
        test_worked_example_golden,
        test_single_key_row_is_exact,
        test_zero_keys_give_prefix_mean,
        test_peaked_scores_pick_the_argmax_value,
        lambda: test_forward_matches_scalar_brute_force(True, 2, 2, 7, 8),
        lambda: test_forward_matches_scalar_brute_force(False, 2, 2, 7, 8),
        lambda: test_backward_sum_invariants(True),
    ]
    for chk in checks:
        try:
            chk()
        except AssertionError:
            return False
    return True


def test_pins_pass_on_the_real_oracle():
    assert _pins_pass()


_REAL_SOFTMAX = oatt._softmax_rows


def _mut_visible_strict(rows, n_keys, causal):
    j = np.arange(n_keys)
    if causal:
        return j[None, :] < np.asarray(rows)[:, None]   # diagonal dropped
    return np.ones((len(rows), n_keys), dtype=bool)


def _mut_visible_transposed(rows, n_keys, causal):
    j = np.arange(n_keys)
    if causal:
        return j[None, :] >= np.asarray(rows)[:, None]  # future keys instead of past
    return np.ones((len(rows), n_keys), dtype=bool)


def _mut_softmax_lse_drops_max(s, vis):
    p, lse = _REAL_SOFTMAX(s, vis)
    m = np.where(vis, s, -np.inf).max(axis=1)
    return p, lse - np.where(np.isfinite(m), m, 0.0)


def _mut_softmax_unnormalised(s, vis):
    p, lse = _REAL_SOFTMAX(s, vis)
    return p * 1.0001, lse


def _mut_bwd(field, how):
    real_bwd = oatt.attn_bwd

    def bwd(*a, **kw):
        r = real_bwd(*a, **kw)
        r[field] = how(r[field])
        return r
    return bwd


@pytest.mark.parametrize("mutation", ["mask_strict", "mask_transposed", "lse_drops_max", "unnormalised",
                                      "dk_sign", "dv_keys_reversed", "dq_unscaled"])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    if mutation == "mask_strict":
        monkeypatch.setattr(oatt, "_visible", _mut_visible_strict)
    elif mutation == "mask_transposed":
        monkeypatch.setattr(oatt, "_visible", _mut_visible_transposed)
    elif mutation == "lse_drops_max":
        monkeypatch.setattr(oatt, "_softmax_rows", _mut_softmax_lse_drops_max)
    elif mutation == "unnormalised":
        monkeypatch.setattr(oatt, "_softmax_rows", _mut_softmax_unnormalised)
    else:
        field, how = {
            "dk_sign": ("dk", lambda x: -x),
            "dv_keys_reversed": ("dv", lambda x: x[:, ::-1].copy()),
            "dq_unscaled": ("dq", lambda x: 2.0 * x),
        }[mutation]
        monkeypatch.setattr(oracle, "attn_bwd", _mut_bwd(field, how))
    assert not _pins_pass(), f"planted mistake {mutation} went unnoticed"


# ---------------------------------------------------------------- RoPE

def _rope_scalar(x, theta, pos0, inverse=False):
    """RoPE by plain scalar loops with math.cos / math.sin (tiny inputs only)."""
    B, S, H, D = x.shape
    half = D // 2
    y = np.zeros_like(x, dtype=np.float64)
    for b in range(B):
        for i in range(S):
            for h in range(H):
                for k in range(half):
                    a = (pos0 + i) * theta ** (-2.0 * k / D)
                    if inverse:
                        a = -a
                    lo, hi = float(x[b, i, h, k]), float(x[b, i, h, k + half])
                    y[b, i, h, k] = lo * math.cos(a) - hi * math.sin(a)
                    y[b, i, h, k + half] = hi * math.cos(a) + lo * math.sin(a)
    return y


def test_rope_matches_scalar_loops():
    rng = np.random.default_rng(61)
    x = rng.standard_normal((2, 5, 2, 8))
    for theta, pos0 in ((1e4, 0), (1e6, 524283), (1e9, 17)):
        for inv in (False, True):
            np.testing.assert_allclose(oracle.rope(x, theta, pos0, inv), _rope_scalar(x, theta, pos0, inv),
                                       atol=1e-12, rtol=0)


def test_rope_closed_forms():
    # D = 4, theta = 100: pair 0 turns by i radians, pair 1 by i / 10; features (0, 2) and (1, 3) pair up
    x = np.zeros((1, 3, 1, 4))
    x[0, :, 0, 0] = 1.0   # unit vector in pair 0
    x[0, :, 0, 3] = 2.0   # second feature of pair 1
    y = oracle.rope(x, 100.0)
    for i in range(3):
        assert y[0, i, 0, 0] == pytest.approx(math.cos(i), abs=1e-15)
        assert y[0, i, 0, 2] == pytest.approx(math.sin(i), abs=1e-15)
        assert y[0, i, 0, 1] == pytest.approx(-2.0 * math.sin(i / 10), abs=1e-15)
        assert y[0, i, 0, 3] == pytest.approx(2.0 * math.cos(i / 10), abs=1e-15)
    # position 0 is the identity, exactly
    rng = np.random.default_rng(62)
    z = rng.standard_normal((1, 1, 3, 16))
    assert np.array_equal(oracle.rope(z, 1e6), z)


def test_rope_invariants():
    rng = np.random.default_rng(63)
    q = rng.standard_normal((1, 6, 2, 16))
    k = rng.standard_normal((1, 6, 2, 16))
    yq = oracle.rope(q, 1e6, 1000)
    # each pair keeps its length; the inverse undoes the rotation
    n0 = q[..., :8] ** 2 + q[..., 8:] ** 2
    n1 = yq[..., :8] ** 2 + yq[..., 8:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12)
    np.testing.assert_allclose(oracle.rope(yq, 1e6, 1000, inverse=True), q, atol=1e-12)
    # scores depend on positions only through their difference: shifting every position keeps q_i . k_j
    s1 = np.einsum("bihd,bjhd->bhij", oracle.rope(q, 1e6, 0), oracle.rope(k, 1e6, 0))
    s2 = np.einsum("bihd,bjhd->bhij", oracle.rope(q, 1e6, 77777), oracle.rope(k, 1e6, 77777))
    np.testing.assert_allclose(s2, s1, atol=1e-10)


def test_planted_rope_mistakes_are_caught():
    """Interleaved pairs (2k, 2k+1) or the angle's sign flipped must fail the scalar pin."""
    rng = np.random.default_rng(64)
    x = rng.standard_normal((1, 4, 1, 8))
    want = _rope_scalar(x, 1e4, 3)

    def interleaved(x, theta, pos0):
        y = np.array(x, dtype=np.float64)
        D = x.shape[3]
        for i in range(x.shape[1]):
            for k in range(D // 2):
                a = (pos0 + i) * theta ** (-2.0 * k / D)
                lo, hi = x[0, i, 0, 2 * k], x[0, i, 0, 2 * k + 1]
                y[0, i, 0, 2 * k] = lo * math.cos(a) - hi * math.sin(a)
                y[0, i, 0, 2 * k + 1] = hi * math.cos(a) + lo * math.sin(a)
        return y
    assert not np.allclose(interleaved(x, 1e4, 3), want, atol=1e-6)
    assert not np.allclose(oracle.rope(x, 1e4, 3, inverse=True), want, atol=1e-6)
    np.testing.assert_allclose(oracle.rope(x, 1e4, 3), want, atol=1e-12)


# ---------------------------------------------------------------- cross-entropy

def test_ce_matches_scalar_loops():
    rng = np.random.default_rng(71)
    x = rng.standard_normal((4, 7)) * 3
    y = np.array([0, 6, -100, 3])
    loss, lse = oracle.ce_fwd(x, y)
    g = np.array([1.0, 0.5, 2.0, -1.0])
    grad = oracle.ce_grad(x, y, g)
    for i in range(4):
        z = sum(math.exp(v) for v in x[i])
        assert lse[i] == pytest.approx(math.log(z), abs=1e-12)
        if y[i] == -100:
            assert loss[i] == 0.0 and (grad[i] == 0).all()
            continue
        assert loss[i] == pytest.approx(-math.log(math.exp(x[i, y[i]]) / z), abs=1e-12)
        for j in range(7):
            want = g[i] * (math.exp(x[i, j]) / z - (1.0 if j == y[i] else 0.0))
            assert grad[i, j] == pytest.approx(want, abs=1e-12)


def test_ce_closed_forms_and_invariants():
    V = 1000
    x = np.zeros((3, V))
    loss, lse = oracle.ce_fwd(x, [0, 5, 999])
    np.testing.assert_allclose(loss, np.log(V), rtol=1e-14)          # uniform logits: loss = ln V
    x[1, 5] = 80.0
    loss, _ = oracle.ce_fwd(x, [0, 5, 999])
    assert loss[1] < 1e-30                                            # a dominant correct logit: loss -> 0
    rng = np.random.default_rng(72)
    z = rng.standard_normal((5, 50)) * 4
    y = rng.integers(0, 50, 5)
    grad = oracle.ce_grad(z, y, 1.0)
    np.testing.assert_allclose(grad.sum(axis=1), 0.0, atol=1e-13)     # rows of (softmax - onehot) sum to 0
    l1, _ = oracle.ce_fwd(z, y)
    l2, _ = oracle.ce_fwd(z + 123.0, y)                                # a constant per row changes nothing
    np.testing.assert_allclose(l2, l1, atol=1e-11)
    np.testing.assert_allclose(oracle.ce_grad(z + 123.0, y, 1.0), grad, atol=1e-13)


def test_ce_gradient_by_finite_differences():
    rng = np.random.default_rng(73)
    x = rng.standard_normal((3, 9))
    y = np.array([2, -100, 8])
    g = np.array([0.7, 1.3, -0.4])
    grad = oracle.ce_grad(x, y, g)
    h = 1e-6
    for i in range(3):
        for j in range(9):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fd = (np.dot(g, oracle.ce_fwd(xp, y)[0]) - np.dot(g, oracle.ce_fwd(xm, y)[0])) / (2 * h)
            assert grad[i, j] == pytest.approx(fd, abs=1e-8)


def test_planted_ce_mistakes_are_caught():
    """A gradient without the one-hot term, or a loss with the wrong sign, must fail."""
    rng = np.random.default_rng(74)
    x = rng.standard_normal((2, 6))
    y = np.array([1, 4])
    p = np.exp(x - oracle.ce_lse(x)[:, None])
    assert not np.allclose(p, oracle.ce_grad(x, y, 1.0), atol=1e-3)
    loss, lse = oracle.ce_fwd(x, y)
    assert not np.allclose(x[[0, 1], y] - lse, loss, atol=1e-3)


# ---------------------------------------------------------------- Ulysses all-to-all

def test_ulysses_golden_s4_h4_p2():
    """Where every (row, head) lands after the all-to-all, derived by hand."""
    g = _read_golden("ulysses_s4_h4_p2.txt")
    S, H, P, n = 4, 4, 2, 2
    x = np.zeros((1, S, H, 1))
    for s in range(S):
        for h in range(H):
            x[0, s, h, 0] = 10 * s + h  # a distinct tag per (row, head)
    parts = oracle.ulysses_seq_to_head(x, P)
    assert len(g["map"]) == P * S * (H // P)
    for j, s, hh, r, sl, h in ([int(t) for t in toks] for toks in g["map"]):
        assert s == r * n + sl  # the row came from rank r's piece
        assert parts[j][0, s, hh, 0] == 10 * s + h


@pytest.mark.parametrize("B,S,H,D,P", [(1, 8, 4, 3, 2), (2, 12, 6, 2, 3), (1, 16, 8, 4, 8), (2, 6, 5, 2, 1)])
def test_ulysses_round_trip_and_block_sizes(B, S, H, D, P):
    rng = np.random.default_rng(S * H + P)
    x = rng.standard_normal((B, S, H, D))
    parts = oracle.ulysses_seq_to_head(x, P)
    assert all(p.shape == (B, S, H // P, D) for p in parts)
    # rank j holds all rows of head group j and nothing else
    for j, p in enumerate(parts):
        assert np.array_equal(p, x[:, :, j * (H // P):(j + 1) * (H // P)])
    assert np.array_equal(oracle.ulysses_head_to_seq(parts, P), x)
    bad = np.zeros((1, S + 1, H, D)) if P > 1 else np.zeros((1, S, H, D))
    with pytest.raises(ValueError):  # a sequence P does not divide, or no ranks
        oracle.ulysses_seq_to_head(bad, P if P > 1 else 0)


@pytest.mark.parametrize("causal", [True, False])
def test_ulysses_attention_equals_monolithic(causal):
    rng = np.random.default_rng(7)
    B, S, H, D, P = 2, 12, 6, 4, 3
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    o, lse = oracle.ulysses_attn_fwd(q, k, v, P, causal, 0.5)
    om, lsem = oracle.attn_fwd(q, k, v, causal, 0.5)
    np.testing.assert_allclose(o, om, atol=1e-13)
    np.testing.assert_allclose(lse, lsem, atol=1e-13)


def test_ulysses_pins_catch_a_transposed_exchange(monkeypatch):
    """A planted mistake: the receiving rank takes head group r (the sender's
    index) instead of its own j. The golden map must fail."""
    import oracle.ulysses as oul

    def wrong(x, P):
        B, S, H, D = x.shape
        n, hp = S // P, H // P
        out = [np.empty((B, S, hp, D)) for _ in range(P)]
        for r in range(P):
            for j in range(P):
                out[j][:, r * n:(r + 1) * n] = x[:, r * n:(r + 1) * n, r * hp:(r + 1) * hp]
        return out

    monkeypatch.setattr(oracle, "ulysses_seq_to_head", wrong)
    monkeypatch.setattr(oul, "seq_to_head", wrong)
    with pytest.raises(AssertionError):
        test_ulysses_golden_s4_h4_p2()


# ---------------------------------------------------------------- plain (contiguous) ring

def test_ring_golden_s6_p3():
    g = _read_golden("ring_s6_p3.txt")
    perm, tasks = oracle.ring_schedule(6, 3)
    assert [int(x) for x in g["perm"][0]] == list(perm)
    got = sorted((t["rank"], t["step"], t["src"], t["kind"], t["q_off"], t["q_len"], t["k_off"], t["k_len"],
                  t["causal"]) for t in tasks)
    assert got == sorted(tuple(int(x) for x in toks) for toks in g["task"])


def _pairs_per_rank(S, perm, tasks, P):
    per = np.zeros(P, dtype=np.int64)
    for t in tasks:
        one = {**t}
        per[t["rank"]] += oracle.zigzag_tasks_pairs(S, perm, [one]).sum()
    return per


@pytest.mark.parametrize("P,n", [(1, 4), (2, 3), (3, 2), (4, 4), (8, 2)])
def test_ring_covers_every_causal_pair_once_with_rank_imbalance(P, n):
    S = P * n
    perm, tasks = oracle.ring_schedule(S, P)
    count = oracle.zigzag_tasks_pairs(S, perm, tasks)
    want = np.tril(np.ones((S, S), dtype=np.int64))
    assert np.array_equal(count, want)  # every causal pair exactly once
    per = _pairs_per_rank(S, perm, tasks, P)
    # rank r: one causal block and r full blocks
    assert list(per) == [n * (n + 1) // 2 + r * n * n for r in range(P)]
    assert per.sum() == S * (S + 1) // 2
    # the zigzag split of the same sequence (when it exists) gives every rank the same count
    if S % (2 * P) == 0:
        zperm, ztasks = oracle.zigzag_schedule(S, P)
        zper = _pairs_per_rank(S, zperm, ztasks, P)
        assert len(set(zper.tolist())) == 1 and zper.sum() == per.sum()
    for t in tasks:  # a NONE task has no work, and only later ranks' keys give NONE
        if t["kind"] == oracle.TASK_NONE:
            assert t["q_len"] == 0 and t["k_len"] == 0 and t["src"] > t["rank"]


def test_ring_rejects_bad_sizes():
    for S, P in ((7, 2), (0, 1), (4, 0), (3, 4)):
        with pytest.raises(ValueError):
            oracle.ring_schedule(S, P)
