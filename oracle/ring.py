"""Ring attention as the pages state it: shards, schedule, the loop, work.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Shard layouts (which global token positions a rank owns, in local order):
  * contiguous - the tutorial "06 - Sequence / Context Parallelism",
    section 1 diagram: GPU k holds tokens [k*S/c, (k+1)*S/c);
  * zig-zag - the plate "Splitting the Sequence": the sequence is cut into
    2c chunks and device k gets chunks k and 2c-1-k (also its "Terms" list).
    Reading: k counts from 0 (counting from 1 would leave chunk 2c unowned);
    the two chunks are concatenated in increasing position.
  * striped - the tutorial's section 5 ("striped / zigzag attention":
    tokens assigned to GPUs in an interleaved pattern; section 12 cites
    Striped Attention).  Reading: round robin, rank k owns every token whose
    position is k mod c, in increasing position.

Ring schedule (tutorial section 4): every rank sends its held K/V to rank
i+1 and receives from i-1 after each step, so at step t rank i holds the
block that started on rank (i - t) mod c.  Reading: c compute steps (the
tutorial loops N times; the plate's "c - 1 passes" counts transfers).

The loop (tutorial section 4): out, m, l = initialise(); for each step,
attend Q_i to the held block and update (out, m, l) with online-softmax
rescaling; finally out / l.

Work (tutorial section 10 exercise B; plate "One sequence, sixteen
devices": at c = 16 the busiest contiguous device does 1.94x the average;
zig-zag makes the work equal): counted here by direct summation over
(query, key) pairs and over 128x128 tiles, never from a closed form.
"""

from __future__ import annotations

import numpy as np


CONTIGUOUS = "contiguous"
ZIGZAG = "zigzag"
STRIPED = "striped"


def shard_positions(S, c, layout):
    """Global positions owned by each of the c ranks, in local order."""
    if layout == CONTIGUOUS:
        if S % c:
            raise ValueError("contiguous split needs S divisible by c")
        n = S // c
        return [np.arange(r * n, (r + 1) * n, dtype=np.int64) for r in range(c)]
    if layout == ZIGZAG:
        if S % (2 * c):
            raise ValueError("zig-zag split needs S divisible by 2c")
        ch = S // (2 * c)
        return [np.concatenate([np.arange(r * ch, (r + 1) * ch),
                                np.arange((2 * c - 1 - r) * ch, (2 * c - r) * ch)]).astype(np.int64)
                for r in range(c)]
    if layout == STRIPED:
        if S % c:
            raise ValueError("striped split needs S divisible by c")
        return [np.arange(r, S, c, dtype=np.int64) for r in range(c)]
    raise ValueError(f"unknown layout {layout!r}")


def ring_source(i, t, c):
    """Rank whose K/V block rank i holds at step t (send to i+1, receive from i-1)."""
    return (i - t) % c


def schedule(c):
    """c x c table: schedule[t][i] = source rank of the block rank i attends at step t."""
    return [[ring_source(i, t, c) for i in range(c)] for t in range(c)]


def block_partial(qi, kb, vb, qp, kp, causal, scale):
    """Attention of a query block to one key/value block, unnormalised.

    Returns (o [B,n,Hq,D], m [B,Hq,n], l [B,Hq,n]): the block max of the
    scaled visible scores, the sum of exp(s - m) and the exp-weighted sum of
    values.  Rows with no visible key give m = -inf, l = 0, o = 0.
    """
    B, n, Hq, D = qi.shape
    Hkv = kb.shape[2]
    G = Hq // Hkv
    o = np.zeros((B, n, Hq, D))
    m = np.full((B, Hq, n), -np.inf)
    l = np.zeros((B, Hq, n))
    if causal:
        vis = np.asarray(kp)[None, :] <= np.asarray(qp)[:, None]
    else:
        vis = np.ones((n, kb.shape[1]), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            s = scale * (qi[b, :, h, :] @ kb[b, :, g, :].T)
            s = np.where(vis, s, -np.inf)
            mb = s.max(axis=1) if s.shape[1] else np.full(n, -np.inf)
            shift = np.where(np.isfinite(mb), mb, 0.0)
            e = np.where(vis, np.exp(s - shift[:, None]), 0.0)
            m[b, h] = mb
            l[b, h] = e.sum(axis=1)
            o[b, :, h, :] = e @ vb[b, :, g, :]
    return o, m, l


def ring_attention(q, k, v, c, layout, causal, scale, order=None):
    """The ring loop in float64, one virtual rank after another.

    q: [B, S, Hq, D]; k, v: [B, S, Hkv, D] in natural token order.  For each
    rank i: initialise (out = 0, m = -inf, l = 0); for each step t attend the
    rank's queries to the block of rank (i - t) mod c (or of ``order[i][t]``
    when an explicit block order is given, to check that any order gives the
    same answer) and fold the block in with online-softmax rescaling; finally
    divide by l.  Returns (out [B,S,Hq,D], lse [B,Hq,S]) in natural order.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, S, Hq, D = q.shape
    shards = shard_positions(S, c, layout)
    out_full = np.zeros((B, S, Hq, D))
    lse_full = np.full((B, Hq, S), -np.inf)
    for i in range(c):
        qp = shards[i]
        qi = q[:, qp]
        n = qp.shape[0]
        # initialise(): the online-softmax state of rank i
        o = np.zeros((B, n, Hq, D))
        m = np.full((B, Hq, n), -np.inf)
        l = np.zeros((B, Hq, n))
        steps = order[i] if order is not None else [ring_source(i, t, c) for t in range(c)]
        for j in steps:
            kp = shards[j]
            # partial attention of Q_i against the held block
            ob, mb, lb = block_partial(qi, k[:, kp], v[:, kp], qp, kp, causal, scale)
            # update with rescaling: earlier sums are scaled by exp(m - m_new)
            m_new = np.maximum(m, mb)
            safe = np.where(np.isfinite(m_new), m_new, 0.0)
            a_old = np.where(np.isfinite(m), np.exp(m - safe), 0.0)
            a_blk = np.where(np.isfinite(mb), np.exp(mb - safe), 0.0)
            l = l * a_old + lb * a_blk
            o = (o * np.transpose(a_old, (0, 2, 1))[..., None]
                 + ob * np.transpose(a_blk, (0, 2, 1))[..., None])
            m = m_new
        # out_i = out_i / l_i
        pos = l > 0
        ls = np.where(pos, l, 1.0)
        out_full[:, qp] = np.where(np.transpose(pos, (0, 2, 1))[..., None],
                                   o / np.transpose(ls, (0, 2, 1))[..., None], 0.0)
        with np.errstate(divide="ignore"):
            lse_full[:, :, qp] = np.where(pos, m + np.log(ls), -np.inf)
    return out_full, lse_full


def allgather_attention(q, k, v, c, layout, causal, scale):
    """The all-gather form of context parallelism in float64.

    The plate "Splitting the Sequence" notes that Llama 3 gathers every
    rank's keys and values instead of passing them round a ring.  Each rank
    first collects all c shards (in rank order), then attends its queries to
    the gathered keys once, with the causal mask by global position.
    Returns (out [B,S,Hq,D], lse [B,Hq,S]) in natural order.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, S, Hq, D = q.shape
    shards = shard_positions(S, c, layout)
    gathered = np.concatenate(shards)                # all-gather: every shard, rank order
    out_full = np.zeros((B, S, Hq, D))
    lse_full = np.full((B, Hq, S), -np.inf)
    for i in range(c):
        qp = shards[i]
        o, m, l = block_partial(q[:, qp], k[:, gathered], v[:, gathered], qp, gathered, causal, scale)
        pos = l > 0
        ls = np.where(pos, l, 1.0)
        out_full[:, qp] = np.where(np.transpose(pos, (0, 2, 1))[..., None],
                                   o / np.transpose(ls, (0, 2, 1))[..., None], 0.0)
        with np.errstate(divide="ignore"):
            lse_full[:, :, qp] = np.where(pos, m + np.log(ls), -np.inf)
    return out_full, lse_full


def decode_split_kv(q_new, q_pos, k, v, c, layout, causal, scale):
    """Attention of a few new queries over keys and values spread over c
    shards, in float64: every shard computes its partial state for the
    queries (split over the keys), and the partials are gathered and merged
    (the tutorial's section 7: decode over distributed keys and values needs a
    gather of partial results, like a split-K).  q_new: [B, R, Hq, D];
    q_pos: [R] global positions.  Returns (out [B,R,Hq,D], lse [B,Hq,R]) and
    the per-shard partials (o, m, l) that were merged."""
    from .merge import finalize_state, merge_states

    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S = k.shape[1]
    parts = []
    for kp in shard_positions(S, c, layout):
        parts.append(block_partial(np.asarray(q_new, dtype=np.float64), k[:, kp], v[:, kp],
                                   np.asarray(q_pos), kp, causal, scale))
    O, M, L = merge_states([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts])
    out, lse = finalize_state(O, M, L)
    return out, lse, parts


def visible_pairs(qp, kp, causal):
    """Number of (query, key) pairs with k_pos <= q_pos (all pairs if not causal)."""
    qp = np.asarray(qp, dtype=np.int64)
    kp = np.asarray(kp, dtype=np.int64)
    if not causal:
        return int(qp.size) * int(kp.size)
    ks = np.sort(kp)
    return int(np.searchsorted(ks, qp, side="right").sum())


def tile_classes(qp, kp, causal, tile=128):
    """Classify every (query tile, key tile) pair of one (rank, step) block.

    Tiles are runs of ``tile`` rows of each shard's local order (the last one
    may be short).  A tile pair is 'skipped' when none of its pairs is
    visible, 'full' when all are, 'partial' otherwise.  The visible pairs of
    each tile pair are counted one query at a time (the number of the key
    tile's positions <= that query's position), so no min/max shortcut is
    used.  Returns (full, partial, skipped).
    """
    qp = np.asarray(qp, dtype=np.int64)
    kp = np.asarray(kp, dtype=np.int64)
    full = partial = skipped = 0
    if qp.size == 0 or kp.size == 0:
        return 0, 0, 0
    starts = np.arange(0, qp.size, tile)
    qsize = np.diff(np.append(starts, qp.size))
    for b in range(0, kp.size, tile):
        kt = np.sort(kp[b:b + tile])
        if causal:
            per_query = np.searchsorted(kt, qp, side="right")
        else:
            per_query = np.full(qp.size, kt.size)
        vis = np.add.reduceat(per_query, starts)
        total = qsize * kt.size
        skipped += int((vis == 0).sum())
        full += int((vis == total).sum())
        partial += int(((vis > 0) & (vis < total)).sum())
    return full, partial, skipped


def work_table(S, c, layout, causal, tile=128):
    """Per (rank, step) work of one (batch, head): dict with arrays [c, c]
    'pairs', 'full', 'partial', 'skipped', indexed [rank][step]."""
    shards = shard_positions(S, c, layout)
    out = {key: np.zeros((c, c), dtype=np.int64) for key in ("pairs", "full", "partial", "skipped")}
    for i in range(c):
        for t in range(c):
            j = ring_source(i, t, c)
            out["pairs"][i, t] = visible_pairs(shards[i], shards[j], causal)
            f, p, s = tile_classes(shards[i], shards[j], causal, tile)
            out["full"][i, t] = f
            out["partial"][i, t] = p
            out["skipped"][i, t] = s
    return out


def imbalance(per_rank_work):
    """Busiest rank's work over the mean (every rank waits for the busiest)."""
    w = np.asarray(per_rank_work, dtype=np.float64)
    return float(w.max() / w.mean())


def ring_kv_bytes(S, Hkv, D, elem_bytes, B=1, c=None):
    """K/V bytes one layer's ring moves per device.

    Tutorial section 4: every step each device sends its K and V once, so
    over N steps it moves N * (S/N) * n_kv_heads * head_dim * 2 * bytes, which
    is S * n_kv_heads * head_dim * 2 * bytes whatever N is.  With ``c`` given,
    the plate's form: (c - 1)/c of that (the device's own block is not sent).
    """
    full = S * Hkv * D * 2 * elem_bytes * B
    if c is None:
        return full
    return full * (c - 1) // c
