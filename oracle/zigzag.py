"""Oracle for the zigzag ring split and its per-(rank, step) attention tasks.

TEST INFRASTRUCTURE (see the package header).

Zigzag ring attention ("EasyContext代码解析200行核心训练脚本实现原理",
§模型并行策略解析 "zigzag_ring_attn" and §训练循环核心逻辑, where
prepare_seq_parallel_inputs cuts each sequence into the rank-local pieces)
splits a sequence of S tokens into 2P chunks of c = S / (2P) tokens. Rank r
of P holds chunk r and chunk 2P-1-r, in that order, so that every rank owns
one early and one late chunk and the causal work is equal across ranks.

Zigzag order: the concatenation of the ranks' local sequences, rank 0 first.
perm[t] is the natural (global) token index at zigzag position t.

Ring: at step s (0 <= s < P) rank r holds the keys and values of rank
src = (r - s) mod P (they travel r -> r+1; the opposite direction gives the
same set of tasks). Ordering the chunks shows which (query, key) pairs of
that step are causal-visible:

  s = 0, DIAG : local queries x local keys, causal in local order (chunk r
                precedes chunk 2P-1-r, so local order agrees with global).
  src < r, LOWER: all 2c local queries x src's first chunk (c keys), all
                visible (chunk src precedes both of r's chunks; src's second
                chunk follows both and is seen by none).
  src > r, UPPER: r's second chunk (c queries) x all 2c keys of src, all
                visible (both of src's chunks lie between r's two chunks).

Offsets below are positions in zigzag order.
"""

import numpy as np

TASK_DIAG, TASK_LOWER, TASK_UPPER = 0, 1, 2


def zigzag_schedule(S, P):
    """Returns (perm [S] int64, tasks list of dicts) or raises ValueError."""
    if P < 1 or S < 2 * P or S % (2 * P) != 0:
        raise ValueError("zigzag needs P >= 1 and S a positive multiple of 2P")
    c = S // (2 * P)
    perm = np.empty(S, dtype=np.int64)
    for r in range(P):
        early, late = r, 2 * P - 1 - r
        base = r * 2 * c
        perm[base:base + c] = np.arange(early * c, early * c + c)
        perm[base + c:base + 2 * c] = np.arange(late * c, late * c + c)
    tasks = []
    for r in range(P):
        for s in range(P):
            src = (r - s) % P
            if s == 0:
                kind, q_off, q_len, k_off, k_len, causal = TASK_DIAG, r * 2 * c, 2 * c, r * 2 * c, 2 * c, 1
            elif src < r:
                kind, q_off, q_len, k_off, k_len, causal = TASK_LOWER, r * 2 * c, 2 * c, src * 2 * c, c, 0
            else:
                kind, q_off, q_len, k_off, k_len, causal = TASK_UPPER, r * 2 * c + c, c, src * 2 * c, 2 * c, 0
            tasks.append({"rank": r, "step": s, "src": src, "kind": kind,
                          "q_off": q_off, "q_len": q_len, "k_off": k_off,
                          "k_len": k_len, "causal": causal})
    return perm, tasks


def zigzag_tasks_pairs(S, perm, tasks):
    """Brute force: how many times each global (query, key) pair is computed.

    Returns an int64 [S, S] count matrix (small S only). A correct schedule
    has count 1 on every causal pair (key <= query) and 0 elsewhere.
    """
    count = np.zeros((S, S), dtype=np.int64)
    for t in tasks:
        for a in range(t["q_len"]):
            for b in range(t["k_len"]):
                if t["causal"] and b > a:
                    continue
                count[perm[t["q_off"] + a], perm[t["k_off"] + b]] += 1
    return count


TASK_FULL, TASK_NONE = 3, 4


def ring_schedule(S, P):
    """The plain ring: the contiguous split the zigzag split improves on.

    Rank r holds rows [r S/P, (r+1) S/P) (perm is the identity). At step s it
    holds the keys of src = (r - s) mod P:
      s = 0, DIAG : local queries x local keys, causal;
      src < r, FULL: all local queries x all of src's keys, all visible;
      src > r, NONE: src's keys all follow every local query: no work.
    Rank r does r full blocks and one causal block, so the last rank does
    about 2(P-1)/P times the average work; the zigzag split makes every
    rank's work equal.
    """
    if P < 1 or S < P or S % P != 0:
        raise ValueError("the contiguous ring needs P >= 1 and S a positive multiple of P")
    n = S // P
    perm = np.arange(S, dtype=np.int64)
    tasks = []
    for r in range(P):
        for s in range(P):
            src = (r - s) % P
            if s == 0:
                kind, q_len, k_len, causal = TASK_DIAG, n, n, 1
            elif src < r:
                kind, q_len, k_len, causal = TASK_FULL, n, n, 0
            else:
                kind, q_len, k_len, causal = TASK_NONE, 0, 0, 0
            tasks.append({"rank": r, "step": s, "src": src, "kind": kind, "q_off": r * n, "q_len": q_len,
                          "k_off": src * n, "k_len": k_len, "causal": causal})
    return perm, tasks
