"""Pins for the CPU oracle: it is checked against things other than itself.

Brute force with pure-Python loops, closed forms derived by hand, textbook
special cases, the exactness invariant (any ring order equals full softmax),
and the numbers the pages print.  All CPU-only.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import ring
from oracle.merge import finalize_state, merge_states

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_values.json")


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _lists(a):
    return a.tolist()


# --------------------------------------------------------------------------
# Definition: NumPy oracle vs pure-Python brute force
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("B,Sq,Sk,Hq,Hkv,D", [(1, 5, 7, 2, 1, 3), (2, 6, 6, 4, 2, 4), (1, 9, 4, 3, 3, 2)])
def test_reference_matches_bruteforce(causal, B, Sq, Sk, Hq, Hkv, D):
    rng = np.random.default_rng(B * 100 + Sq * 10 + Hq)
    q, k, v = _rand(rng, B, Sq, Hq, D), _rand(rng, B, Sk, Hkv, D), _rand(rng, B, Sk, Hkv, D)
    # scrambled, non-contiguous global positions (the ring hands out arbitrary sets)
    q_pos = rng.permutation(20)[:Sq]
    k_pos = rng.permutation(20)[:Sk]
    scale = 0.37
    out, lse, _, _ = oracle.attention_reference(q, k, v, q_pos, k_pos, causal, scale)
    bo, bl = oracle.attention_bruteforce(_lists(q), _lists(k), _lists(v), q_pos, k_pos, causal, scale)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    bl = np.array(bl)
    fin = np.isfinite(bl)
    assert (fin == np.isfinite(lse)).all()
    np.testing.assert_allclose(lse[fin], bl[fin], rtol=0, atol=1e-12)


def test_reference_row_subset_equals_full():
    rng = np.random.default_rng(3)
    q, k, v = _rand(rng, 2, 12, 4, 5), _rand(rng, 2, 12, 2, 5), _rand(rng, 2, 12, 2, 5)
    pos = np.arange(12)
    full, lse, _, _ = oracle.attention_reference(q, k, v, pos, pos, True, 0.5)
    rows = np.array([11, 0, 7, 7, 3])
    sub, lse_s, _, _ = oracle.attention_reference(q, k, v, pos, pos, True, 0.5, rows=rows)
    np.testing.assert_allclose(sub, full[:, rows], atol=1e-14)
    np.testing.assert_allclose(lse_s, lse[:, :, rows], atol=1e-14)


# --------------------------------------------------------------------------
# Textbook special cases (closed forms)
# --------------------------------------------------------------------------

def test_constant_values_give_that_constant():
    rng = np.random.default_rng(4)
    q, k = _rand(rng, 1, 16, 2, 8), _rand(rng, 1, 16, 1, 8)
    v = np.full((1, 16, 1, 8), 2.5)
    pos = np.arange(16)
    out, _, _, _ = oracle.attention_reference(q, k, v, pos, pos, True, 1.0)
    np.testing.assert_allclose(out, 2.5, atol=1e-13)


def test_zero_queries_give_causal_prefix_mean():
    rng = np.random.default_rng(5)
    S = 10
    q = np.zeros((1, S, 1, 4))
    k, v = _rand(rng, 1, S, 1, 4), _rand(rng, 1, S, 1, 4)
    pos = np.arange(S)
    out, lse, _, _ = oracle.attention_reference(q, k, v, pos, pos, True, 1.0)
    prefix_mean = np.cumsum(v[0, :, 0, :], axis=0) / np.arange(1, S + 1)[:, None]
    np.testing.assert_allclose(out[0, :, 0, :], prefix_mean, atol=1e-13)
    # all scores are 0, so lse = ln(number of visible keys)
    np.testing.assert_allclose(lse[0, 0], np.log(np.arange(1, S + 1)), atol=1e-13)


def test_first_causal_row_sees_only_itself():
    rng = np.random.default_rng(6)
    q, k, v = _rand(rng, 1, 8, 1, 4), _rand(rng, 1, 8, 1, 4), _rand(rng, 1, 8, 1, 4)
    pos = np.arange(8)
    out, lse, _, _ = oracle.attention_reference(q, k, v, pos, pos, True, 0.7)
    np.testing.assert_allclose(out[0, 0, 0], v[0, 0, 0], atol=1e-14)
    assert abs(lse[0, 0, 0] - 0.7 * float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-13


def test_identical_keys_give_uniform_mean():
    rng = np.random.default_rng(7)
    q = _rand(rng, 1, 6, 2, 4)
    k = np.repeat(_rand(rng, 1, 1, 1, 4), 9, axis=1)
    v = _rand(rng, 1, 9, 1, 4)
    out, _, _, _ = oracle.attention_reference(q, k, v, np.arange(6), np.arange(9), False, 1.3)
    np.testing.assert_allclose(out[0, :, :, :], np.broadcast_to(v[0, :, 0, :].mean(0), (6, 2, 4)), atol=1e-13)


def test_gqa_head_mapping_is_contiguous_groups():
    # kv head g carries the constant value g; query head h must read h // G.
    Hq, Hkv = 8, 2
    rng = np.random.default_rng(8)
    q, k = _rand(rng, 1, 5, Hq, 3), _rand(rng, 1, 5, Hkv, 3)
    v = np.zeros((1, 5, Hkv, 3))
    for g in range(Hkv):
        v[:, :, g, :] = g
    out, _, _, _ = oracle.attention_reference(q, k, v, np.arange(5), np.arange(5), True, 1.0)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, :, h, :], h // (Hq // Hkv), atol=1e-13)


def test_row_without_visible_key():
    q, k, v = np.ones((1, 2, 1, 2)), np.ones((1, 3, 1, 2)), np.ones((1, 3, 1, 2))
    out, lse, m, l = oracle.attention_reference(q, k, v, [0, 5], [1, 2, 3], True, 1.0)
    assert np.all(out[0, 0] == 0) and lse[0, 0, 0] == -np.inf and l[0, 0, 0] == 0
    np.testing.assert_allclose(out[0, 1], 1.0)


def test_scale_enters_as_a_temperature():
    # two keys, scores s0, s1: out = sigmoid(scale*(s1 - s0)) blend of v0, v1
    q = np.array([[[[1.0, 0.0]]]])
    k = np.array([[[[0.0, 0.0]], [[2.0, 0.0]]]])
    v = np.array([[[[1.0, 0.0]], [[0.0, 1.0]]]])
    for scale in (0.25, 1.0, 3.0):
        out, lse, _, _ = oracle.attention_reference(q, k, v, [1], [0, 1], True, scale)
        w1 = 1.0 / (1.0 + math.exp(-2.0 * scale))
        np.testing.assert_allclose(out[0, 0, 0], [1 - w1, w1], atol=1e-14)
        assert abs(lse[0, 0, 0] - math.log(1.0 + math.exp(2.0 * scale))) < 1e-13


# --------------------------------------------------------------------------
# The exactness invariant: any ring order == full softmax
# --------------------------------------------------------------------------

@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("c", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("causal", [True, False])
def test_ring_equals_full_softmax(layout, c, causal):
    S = 48
    if S % (2 * c):
        pytest.skip("zig-zag needs S divisible by 2c")
    rng = np.random.default_rng(c * 7 + causal)
    q, k, v = _rand(rng, 2, S, 4, 6) * 2.0, _rand(rng, 2, S, 2, 6) * 2.0, _rand(rng, 2, S, 2, 6)
    pos = np.arange(S)
    ref, lse_ref, _, _ = oracle.attention_reference(q, k, v, pos, pos, causal, 0.41)
    out, lse = ring.ring_attention(q, k, v, c, layout, causal, 0.41)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)
    # any other visiting order of the blocks gives the same result
    order = [list(rng.permutation(c)) for _ in range(c)]
    out2, lse2 = ring.ring_attention(q, k, v, c, layout, causal, 0.41, order=order)
    np.testing.assert_allclose(out2, ref, atol=1e-12)
    np.testing.assert_allclose(lse2, lse_ref, atol=1e-12)


def test_ring_with_one_rank_is_plain_attention():
    rng = np.random.default_rng(9)
    q, k, v = _rand(rng, 1, 10, 2, 3), _rand(rng, 1, 10, 2, 3), _rand(rng, 1, 10, 2, 3)
    bo, bl = oracle.attention_bruteforce(_lists(q), _lists(k), _lists(v), list(range(10)), list(range(10)), True, 0.8)
    out, lse = ring.ring_attention(q, k, v, 1, "contiguous", True, 0.8)
    np.testing.assert_allclose(out, np.array(bo), atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), atol=1e-12)


def test_ring_rescale_under_huge_logits():
    # logits of O(1e3) arriving in later blocks: a dropped rescale would be off by exp(1e3)
    rng = np.random.default_rng(10)
    S, c = 32, 4
    q, k, v = _rand(rng, 1, S, 2, 4) * 30, _rand(rng, 1, S, 1, 4) * 30, _rand(rng, 1, S, 1, 4)
    k[:, S // 2 + 3] += 50.0
    pos = np.arange(S)
    ref, lse_ref, _, _ = oracle.attention_reference(q, k, v, pos, pos, True, 0.5)
    out, lse = ring.ring_attention(q, k, v, c, "zigzag", True, 0.5)
    np.testing.assert_allclose(out, ref, atol=1e-11)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13, atol=1e-11)


# --------------------------------------------------------------------------
# Merge of partial states
# --------------------------------------------------------------------------

@pytest.mark.parametrize("splits", [[7], [1, 20], [0, 5, 5, 31], [31]])
def test_merge_of_any_key_split_equals_unsplit(splits):
    rng = np.random.default_rng(sum(splits) + 1)
    S = 32
    q, k, v = _rand(rng, 1, S, 2, 4) * 3, _rand(rng, 1, S, 1, 4) * 3, _rand(rng, 1, S, 1, 4)
    pos = np.arange(S)
    ref, lse_ref, _, _ = oracle.attention_reference(q, k, v, pos, pos, True, 0.9)
    edges = [0] + splits + [S]
    outs, ms, ls = [], [], []
    for a, b in zip(edges[:-1], edges[1:]):
        o, m, l = ring.block_partial(q, k[:, a:b], v[:, a:b], pos, pos[a:b], True, 0.9)
        outs.append(o)
        ms.append(m)
        ls.append(l)
    O, M, L = merge_states(outs, ms, ls)
    out, lse = finalize_state(O, M, L)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)


def test_merge_single_partial_is_plain_normalisation():
    rng = np.random.default_rng(12)
    O = _rand(rng, 1, 4, 2, 3)
    M = _rand(rng, 1, 2, 4)
    L = np.abs(_rand(rng, 1, 2, 4)) + 0.1
    O2, M2, L2 = merge_states([O], [M], [L])
    np.testing.assert_allclose(O2, O, atol=0)
    out, lse = finalize_state(O2, M2, L2)
    np.testing.assert_allclose(out, O / np.transpose(L, (0, 2, 1))[..., None], atol=1e-15)
    np.testing.assert_allclose(lse, M + np.log(L), atol=1e-15)


# --------------------------------------------------------------------------
# Layouts and the ring schedule
# --------------------------------------------------------------------------

@pytest.mark.parametrize("c", [1, 2, 4, 16])
def test_layouts_partition_the_sequence(c):
    S = 64 * c
    for layout in ("contiguous", "zigzag", "striped"):
        shards = ring.shard_positions(S, c, layout)
        allpos = np.sort(np.concatenate(shards))
        assert np.array_equal(allpos, np.arange(S))
        assert all(s.size == S // c for s in shards)
    ch = S // (2 * c)
    z = ring.shard_positions(S, c, "zigzag")
    for r in range(c):
        # rank r holds chunks r and 2c-1-r, in increasing order
        assert np.array_equal(z[r][:ch] // ch, np.full(ch, r))
        assert np.array_equal(z[r][ch:] // ch, np.full(ch, 2 * c - 1 - r))
        assert np.all(np.diff(z[r]) > 0)


@pytest.mark.parametrize("c", [1, 2, 3, 5, 16])
def test_schedule_matches_a_literal_send_recv_simulation(c):
    # every rank starts with its own block, sends what it holds to i+1 and
    # receives from i-1 after each step
    held = list(range(c))
    sched = ring.schedule(c)
    seen = [set() for _ in range(c)]
    for t in range(c):
        for i in range(c):
            assert sched[t][i] == held[i]
            seen[i].add(held[i])
        sent = list(held)
        for i in range(c):
            held[(i + 1) % c] = sent[i]
    assert all(s == set(range(c)) for s in seen)


# --------------------------------------------------------------------------
# Work counts: hand-derived closed forms and the pages' printed values
# --------------------------------------------------------------------------

@pytest.mark.parametrize("S,c", [(1024, 4), (4096, 8), (131072, 16)])
def test_contiguous_pair_counts_closed_form(S, c):
    n = S // c
    shards = ring.shard_positions(S, c, "contiguous")
    per_rank = [sum(ring.visible_pairs(shards[i], shards[j], True) for j in range(c)) for i in range(c)]
    # rank r sees r full blocks plus its own causal triangle
    assert per_rank == [r * n * n + n * (n + 1) // 2 for r in range(c)]
    assert abs(ring.imbalance(per_rank) - ((2 * c - 1) * n + 1) / (c * n + 1)) < 1e-15


@pytest.mark.parametrize("S,c", [(64, 4), (4096, 4), (32768, 8), (131072, 16)])
def test_striped_pair_counts_closed_form(S, c):
    # rank k's a-th query sits at position k + c*a and sees k + c*a + 1 keys,
    # so rank k sees c*n(n-1)/2 + n(k+1) pairs: nearly, not exactly, equal
    n = S // c
    shards = ring.shard_positions(S, c, "striped")
    assert all(np.array_equal(shards[k], np.arange(k, S, c)) for k in range(c))
    per_rank = [sum(ring.visible_pairs(shards[i], shards[j], True) for j in range(c)) for i in range(c)]
    assert per_rank == [c * n * (n - 1) // 2 + n * (k + 1) for k in range(c)]
    assert ring.imbalance(per_rank) < 1 + 1.0 / n


@pytest.mark.parametrize("S,c", [(4096, 4), (32768, 8), (131072, 16), (65536, 8)])
def test_zigzag_pair_counts_are_equal(S, c):
    ch = S // (2 * c)
    shards = ring.shard_positions(S, c, "zigzag")
    per_rank = [sum(ring.visible_pairs(shards[i], shards[j], True) for j in range(c)) for i in range(c)]
    assert per_rank == [(2 * c - 1) * ch * ch + ch * (ch + 1)] * c
    assert ring.imbalance(per_rank) == 1.0


def test_pages_printed_imbalance():
    g = json.load(open(GOLDEN))
    e = g["imbalance_contiguous_c16"]
    S, c = e["S"], e["c"]
    shards = ring.shard_positions(S, c, "contiguous")
    per_rank = [sum(ring.visible_pairs(shards[i], shards[j], True) for j in range(c)) for i in range(c)]
    assert round(ring.imbalance(per_rank), e["decimals"]) == e["value"]
    # the area form of the same quantity is exactly 2 - 1/c
    area = [(r + 0.5) for r in range(c)]
    assert ring.imbalance(area) == 2 - 1 / c
    z = ring.shard_positions(S, c, "zigzag")
    zw = [sum(ring.visible_pairs(z[i], z[j], True) for j in range(c)) for i in range(c)]
    assert ring.imbalance(zw) == g["imbalance_zigzag"]["value"]


def test_tile_counts_hand_derived():
    # 32768 tokens, c=8, 128x128 tiles, one head.  Contiguous rank r at step t
    # with source j: j<r all 32x32 tiles full, j==r the causal triangle
    # (496 full, 32 diagonal partial, 496 skipped), j>r all skipped.
    T = 32
    w = ring.work_table(32768, 8, "contiguous", True)
    for r in range(8):
        assert w["full"][r].sum() == T * T * r + T * (T - 1) // 2
        assert w["partial"][r].sum() == T
        assert w["skipped"][r].sum() == T * T * (7 - r) + T * (T - 1) // 2
    # zig-zag (chunks of 2048 = 16 tiles): every foreign step sees exactly two
    # of the four chunk pairs fully (512 full, 512 skipped); its own step has
    # two triangles and one full chunk pair.
    z = ring.work_table(32768, 8, "zigzag", True)
    for r in range(8):
        for t in range(1, 8):
            assert (z["full"][r, t], z["partial"][r, t], z["skipped"][r, t]) == (512, 0, 512)
        assert (z["full"][r, 0], z["partial"][r, 0], z["skipped"][r, 0]) == (2 * 120 + 256, 32, 2 * 120 + 256)


def test_tile_counts_ragged_and_noncausal():
    w = ring.work_table(600, 2, "contiguous", False)
    # 300 rows per rank -> tiles of 128, 128, 44: 3x3 tile pairs, all full
    assert (w["full"] == 9).all() and (w["partial"] == 0).all() and (w["skipped"] == 0).all()
    assert (w["pairs"] == 300 * 300).all()
    # causal: the own block has the triangle only
    wc = ring.work_table(600, 2, "contiguous", True)
    assert wc["pairs"][0, 0] == 300 * 301 // 2 and wc["pairs"][0, 1] == 0
    assert wc["pairs"][1, 1] == 300 * 300


# --------------------------------------------------------------------------
# Derived ring traffic and the plate's 12.7 %
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 2, 4, 8, 16, 64])
def test_ring_volume_independent_of_N(N):
    S, Hkv, D, eb = 131072, 8, 128, 2
    per_step = (S // N) * Hkv * D * 2 * eb    # one block's K and V
    assert N * per_step == ring.ring_kv_bytes(S, Hkv, D, eb)


def test_plate_transfer_to_compute_ratio():
    e = json.load(open(GOLDEN))["ring_transfer_over_compute"]
    S, c, D = e["S"], e["c"], e["head_dim"]
    moved = ring.ring_kv_bytes(S, e["kv_heads_per_device"], D, e["bytes"], c=c)
    assert moved == 62914560
    t_net = moved / (e["network_gbit_s"] * 1e9 / 8)
    pairs = S * S / 2 / c                      # balanced causal work per device
    flop = 4 * pairs * D * e["q_heads_per_device"]
    t_att = flop / (e["attention_efficiency"] * e["external_assumption_h100_dense_bf16_tflops"] * 1e12)
    assert round(t_net / t_att, e["decimals"]) == e["value"]


# --------------------------------------------------------------------------
# All-gather form and decode over distributed keys (next rows)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_allgather_equals_full_softmax(layout):
    rng = np.random.default_rng(21)
    S, c = 48, 4
    q, k, v = _rand(rng, 2, S, 4, 5) * 3, _rand(rng, 2, S, 2, 5) * 3, _rand(rng, 2, S, 2, 5)
    pos = np.arange(S)
    ref, lse_ref, _, _ = oracle.attention_reference(q, k, v, pos, pos, True, 0.6)
    out, lse = ring.allgather_attention(q, k, v, c, layout, True, 0.6)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_decode_split_kv_equals_full_softmax(layout):
    rng = np.random.default_rng(22)
    S, c, R = 64, 4, 3
    k, v = _rand(rng, 1, S, 2, 6) * 2, _rand(rng, 1, S, 2, 6)
    q_new = _rand(rng, 1, R, 8, 6) * 2
    q_pos = np.array([S - 1, 40, 5])              # the newest token and two earlier ones
    ref, lse_ref, _, _ = oracle.attention_reference(q_new, k, v, q_pos, np.arange(S), True, 0.4)
    out, lse, parts = ring.decode_split_kv(q_new, q_pos, k, v, c, layout, True, 0.4)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)
    assert len(parts) == c
