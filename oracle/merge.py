"""Combination of partial online-softmax states, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

A partial state over a key subset K_p is (o_p, m_p, l_p) with
m_p = max_{j in K_p} s_j, l_p = sum_{j in K_p} exp(s_j - m_p) and
o_p = sum_{j in K_p} exp(s_j - m_p) v_j (unnormalised).  Over the disjoint
union of the subsets the same quantities are

    M = max_p m_p,   L = sum_p l_p exp(m_p - M),   O = sum_p o_p exp(m_p - M)

and the attention output is O / L with lse = M + ln L.  This is the rescaling
the quiz "Sequence Parallelism and Ring Attention" (questions 3 and 7)
describes and the final division of the tutorial "06 - Sequence / Context
Parallelism", section 4; the tutorial's section 7 names the same combination
of partial results for decode over distributed keys and values.

m is in natural-log units here.  Partials with m_p = -inf (no key seen)
contribute nothing.
"""

from __future__ import annotations

import numpy as np


def merge_states(outs, ms, ls):
    """Merge P partial states.

    outs: list of [B, S, H, D] unnormalised accumulators; ms, ls: lists of
    [B, H, S].  Returns the merged unnormalised (O [B,S,H,D], M [B,H,S],
    L [B,H,S]).
    """
    ms = [np.asarray(m, dtype=np.float64) for m in ms]
    ls = [np.asarray(l, dtype=np.float64) for l in ls]
    outs = [np.asarray(o, dtype=np.float64) for o in outs]
    M = np.full_like(ms[0], -np.inf)
    for m in ms:
        M = np.maximum(M, m)
    finite = np.isfinite(M)
    Msafe = np.where(finite, M, 0.0)
    L = np.zeros_like(ls[0])
    O = np.zeros_like(outs[0])
    for o, m, l in zip(outs, ms, ls):
        w = np.where(np.isfinite(m), np.exp(m - Msafe), 0.0)   # [B,H,S]
        L = L + l * w
        O = O + o * np.transpose(w, (0, 2, 1))[..., None]
    return O, M, L


def finalize_state(O, M, L):
    """out = O / L, lse = M + ln L; rows with L = 0 give out = 0, lse = -inf."""
    O = np.asarray(O, dtype=np.float64)
    M = np.asarray(M, dtype=np.float64)
    L = np.asarray(L, dtype=np.float64)
    pos = L > 0
    Ls = np.where(pos, L, 1.0)
    out = np.where(np.transpose(pos, (0, 2, 1))[..., None],
                   O / np.transpose(Ls, (0, 2, 1))[..., None], 0.0)
    with np.errstate(divide="ignore"):
        lse = np.where(pos, M + np.log(Ls), -np.inf)
    return out, lse
