"""The definition of exact (causal, grouped-query) softmax attention, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the ring method must reproduce exactly: the tutorial "06 - Sequence /
Context Parallelism", section 4, says the result after the ring is exact, and
its section 10 exercise A asks that it match single-GPU attention; the quiz
"Sequence Parallelism and Ring Attention", question 3, says the blocks are
combined without approximating the full attention pattern.  So the oracle is
single-device softmax attention written out:

    s_ij   = scale * sum_d q[b,i,h,d] * k[b,j,g,d]        g = h // (Hq/Hkv)
    V(i)   = { j : k_pos[j] <= q_pos[i] }  (causal)  or all j
    m_i    = max_{j in V(i)} s_ij
    l_i    = sum_{j in V(i)} exp(s_ij - m_i)
    out_i  = sum_{j in V(i)} exp(s_ij - m_i) v[b,j,g,:] / l_i
    lse_i  = m_i + ln l_i

Readings where the pages are silent:
  * the causal mask compares global token positions and is inclusive (a query
    sees its own key) - the quiz (questions 6, 8) and the plate only say that
    later tokens attend to earlier ones;
  * the softmax scale is an explicit argument (the pages never mention one;
    callers pass 1/sqrt(D));
  * grouped-query heads map in contiguous groups, kv head = h // G (the plate
    gives 8 KV heads for 128 query heads but no mapping);
  * a row that sees no key has m = -inf, l = 0, out = 0, lse = -inf.
"""

from __future__ import annotations

import math

import numpy as np


def _as_f64(x):
    return np.asarray(x, dtype=np.float64)


def attention_reference(q, k, v, q_pos, k_pos, causal, scale, rows=None):
    """Full-row masked softmax attention in float64.

    q: [B, Sq, Hq, D]; k, v: [B, Sk, Hkv, D]; q_pos: [Sq], k_pos: [Sk] integer
    global positions; rows: optional index array into the Sq query rows (the
    result then has R = len(rows) rows in that order).

    Every score of each selected row is materialised, the mask is an explicit
    boolean matrix, and the maximum is subtracted before exponentiating.

    Returns (out [B, R, Hq, D], lse [B, Hq, R], m [B, Hq, R], l [B, Hq, R]),
    with m and lse in natural-log units of the scaled score.
    """
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    B, Sq, Hq, D = q.shape
    Hkv = k.shape[2]
    if Hq % Hkv:
        raise ValueError("query heads must be a multiple of key/value heads")
    G = Hq // Hkv
    if rows is None:
        rows = np.arange(Sq)
    rows = np.asarray(rows, dtype=np.int64)
    R = rows.shape[0]
    out = np.zeros((B, R, Hq, D))
    lse = np.full((B, Hq, R), -np.inf)
    m_all = np.full((B, Hq, R), -np.inf)
    l_all = np.zeros((B, Hq, R))
    if R == 0 or k.shape[1] == 0:
        return out, lse, m_all, l_all
    if causal:
        visible = k_pos[None, :] <= q_pos[rows][:, None]          # [R, Sk]
    else:
        visible = np.ones((R, k.shape[1]), dtype=bool)
    any_visible = visible.any(axis=1)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            scores = scale * (q[b, rows, h, :] @ k[b, :, g, :].T)  # [R, Sk]
            masked = np.where(visible, scores, -np.inf)
            m = masked.max(axis=1)
            shift = np.where(any_visible, m, 0.0)
            e = np.where(visible, np.exp(masked - shift[:, None]), 0.0)
            l = e.sum(axis=1)
            num = e @ v[b, :, g, :]
            safe_l = np.where(l > 0, l, 1.0)
            out[b, :, h, :] = np.where(l[:, None] > 0, num / safe_l[:, None], 0.0)
            m_all[b, h] = m
            l_all[b, h] = l
            with np.errstate(divide="ignore"):
                lse[b, h] = np.where(l > 0, m + np.log(safe_l), -np.inf)
    return out, lse, m_all, l_all


def attention_bruteforce(q, k, v, q_pos, k_pos, causal, scale):
    """The same definition with pure-Python loops and math.exp (tiny inputs).

    Written independently of ``attention_reference`` (no NumPy arithmetic) so
    that a slip in one - a transposed operand, a wrong head map, a dropped
    max-shift - shows up as a disagreement.  Returns nested lists
    out[b][i][h][d] and lse[b][h][i].
    """
    B = len(q)
    Sq = len(q[0])
    Hq = len(q[0][0])
    D = len(q[0][0][0])
    Sk = len(k[0])
    Hkv = len(k[0][0])
    G = Hq // Hkv
    out = [[[[0.0] * D for _ in range(Hq)] for _ in range(Sq)] for _ in range(B)]
    lse = [[[float("-inf")] * Sq for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i in range(Sq):
                keys = [j for j in range(Sk)
                        if (not causal) or int(k_pos[j]) <= int(q_pos[i])]
                if not keys:
                    continue
                s = {}
                for j in keys:
                    acc = 0.0
                    for d in range(D):
                        acc += float(q[b][i][h][d]) * float(k[b][j][g][d])
                    s[j] = scale * acc
                mx = max(s.values())
                w = {j: math.exp(s[j] - mx) for j in keys}
                tot = sum(w.values())
                for d in range(D):
                    out[b][i][h][d] = sum(w[j] * float(v[b][j][g][d]) for j in keys) / tot
                lse[b][h][i] = mx + math.log(tot)
    return out, lse
