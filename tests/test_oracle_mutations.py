"""Planted mistakes: each plausible slip in the oracle must fail a pin.

A mutant of ``oracle/attention.py`` is built by editing its source text and
executing it as a fresh module (on the CPU, nothing else changes); the pin
checks below, which depend only on brute force, closed forms and the pages'
statements, must reject every mutant and accept the real oracle.
"""

import inspect
import math
import types

import numpy as np
import pytest

import oracle.attention as real


def _mutant(find, replace):
    src = inspect.getsource(real)
    assert find in src, f"mutation anchor not found: {find!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(find, replace), "<mutant>", "exec"), mod.__dict__)
    return mod


def _pins_hold(mod):
    """True when the module passes every pin check."""
    rng = np.random.default_rng(0)
    checks = []
    # 1. brute force on a GQA case with scrambled positions and large logits
    q = rng.standard_normal((1, 5, 4, 3)) * 8
    k = rng.standard_normal((1, 6, 2, 3)) * 8
    v = rng.standard_normal((1, 6, 2, 3))
    qp, kp = rng.permutation(12)[:5], rng.permutation(12)[:6]
    try:
        with np.errstate(all="ignore"):
            out, lse, _, _ = mod.attention_reference(q, k, v, qp, kp, True, 3.0)
        bo, bl = real.attention_bruteforce(q.tolist(), k.tolist(), v.tolist(), qp, kp, True, 3.0)
        bl = np.array(bl)
        fin = np.isfinite(bl)
        checks.append(np.allclose(out, np.array(bo), atol=1e-9) and
                      (np.isfinite(lse) == fin).all() and np.allclose(lse[fin], bl[fin], atol=1e-9))
    except Exception:
        checks.append(False)
    # 2. Q = 0 gives the causal prefix mean and lse = ln(count)
    S = 7
    q0 = np.zeros((1, S, 1, 2))
    k0, v0 = rng.standard_normal((1, S, 1, 2)), rng.standard_normal((1, S, 1, 2))
    out, lse, _, _ = mod.attention_reference(q0, k0, v0, np.arange(S), np.arange(S), True, 1.0)
    checks.append(np.allclose(out[0, :, 0], np.cumsum(v0[0, :, 0], 0) / np.arange(1, S + 1)[:, None])
                  and np.allclose(lse[0, 0], np.log(np.arange(1, S + 1))))
    # 3. GQA map: kv head g carries the constant g
    v1 = np.zeros((1, 4, 2, 2))
    v1[:, :, 1, :] = 1.0
    out, _, _, _ = mod.attention_reference(rng.standard_normal((1, 4, 4, 2)), rng.standard_normal((1, 4, 2, 2)),
                                           v1, np.arange(4), np.arange(4), True, 1.0)
    checks.append(np.allclose(out[0, :, :2], 0.0) and np.allclose(out[0, :, 2:], 1.0))
    # 4. two keys: the scale acts as a temperature
    qs = np.array([[[[1.0, 0.0]]]])
    ks = np.array([[[[0.0, 0.0]], [[2.0, 0.0]]]])
    vs = np.array([[[[1.0, 0.0]], [[0.0, 1.0]]]])
    out, lse, _, _ = mod.attention_reference(qs, ks, vs, [1], [0, 1], True, 0.25)
    w1 = 1.0 / (1.0 + math.exp(-0.5))
    checks.append(np.allclose(out[0, 0, 0], [1 - w1, w1]) and abs(lse[0, 0, 0] - math.log(1 + math.exp(0.5))) < 1e-12)
    return all(checks)


MUTATIONS = [
    ("g = h // G", "g = h % Hkv"),                                          # wrong head map
    ("k_pos[None, :] <= q_pos[rows][:, None]", "k_pos[None, :] < q_pos[rows][:, None]"),  # strict mask
    ("scores = scale * (q[b, rows, h, :] @ k[b, :, g, :].T)",
     "scores = (q[b, rows, h, :] @ k[b, :, g, :].T)"),                      # dropped scale
    ("np.exp(masked - shift[:, None])", "np.exp(masked)"),                  # dropped max shift
    ("m + np.log(safe_l)", "np.log(safe_l)"),                               # dropped lse term
    ("num / safe_l[:, None]", "num"),                                       # missing normalisation
    ("q[b, rows, h, :] @ k[b, :, g, :].T", "q[b, rows, g, :] @ k[b, :, g, :].T"),  # wrong query head
]


def test_real_oracle_passes_the_pins():
    assert _pins_hold(real)


@pytest.mark.parametrize("find,replace", MUTATIONS)
def test_planted_mistake_is_caught(find, replace):
    assert not _pins_hold(_mutant(find, replace))


# ---------------------------------------------------------------------------
# Mutants of oracle/ring.py: layouts, schedule, the ring update, work counts
# ---------------------------------------------------------------------------

import oracle.ring as real_ring  # noqa: E402


def _ring_mutant(find, replace):
    src = inspect.getsource(real_ring)
    assert find in src, f"mutation anchor not found: {find!r}"
    mod = types.ModuleType("oracle_ring_mutant")
    mod.__dict__["__package__"] = "oracle"
    exec(compile(src.replace(find, replace), "<mutant>", "exec"), mod.__dict__)
    return mod


def _ring_pins_hold(mod):
    checks = []
    # layouts partition the sequence; zig-zag rank r holds chunks r and 2c-1-r
    try:
        S, c = 64, 4
        z = mod.shard_positions(S, c, "zigzag")
        ch = S // (2 * c)
        checks.append(np.array_equal(np.sort(np.concatenate(z)), np.arange(S)) and
                      all(set(z[r] // ch) == {r, 2 * c - 1 - r} for r in range(c)))
    except Exception:
        checks.append(False)
    # schedule equals a literal send-to-(i+1) / receive-from-(i-1) simulation
    c = 5
    held = list(range(c))
    ok = True
    for t in range(c):
        ok &= [mod.ring_source(i, t, c) for i in range(c)] == held
        held = [held[(i - 1) % c] for i in range(c)]
    checks.append(ok)
    # the ring loop equals full softmax (large logits force rescaling)
    rng = np.random.default_rng(1)
    S = 32
    q, k, v = rng.standard_normal((1, S, 2, 4)) * 20, rng.standard_normal((1, S, 1, 4)) * 20, rng.standard_normal((1, S, 1, 4))
    ref, lse_ref, _, _ = real.attention_reference(q, k, v, np.arange(S), np.arange(S), True, 0.5)
    try:
        with np.errstate(all="ignore"):
            out, lse = mod.ring_attention(q, k, v, 4, "zigzag", True, 0.5)
        checks.append(np.allclose(out, ref, atol=1e-9) and np.allclose(lse, lse_ref, atol=1e-9))
    except Exception:
        checks.append(False)
    # hand-derived contiguous pair counts, equal zig-zag work
    S, c = 1024, 4
    n = S // c
    sh = mod.shard_positions(S, c, "contiguous")
    per = [sum(mod.visible_pairs(sh[i], sh[j], True) for j in range(c)) for i in range(c)]
    checks.append(per == [r * n * n + n * (n + 1) // 2 for r in range(c)])
    w = mod.work_table(4096, 8, "contiguous", True)     # 4 tiles of 128 rows per rank
    checks.append(all(w["full"][r].sum() == 16 * r + 6 and w["partial"][r].sum() == 4 for r in range(8)))
    return all(checks)


RING_MUTATIONS = [
    ("np.arange((2 * c - 1 - r) * ch, (2 * c - r) * ch)", "np.arange((2 * c - 2 - r) * ch, (2 * c - 1 - r) * ch)"),
    ("return (i - t) % c", "return (i + t) % c"),
    ("l = l * a_old + lb * a_blk", "l = l + lb * a_blk"),
    ("o = (o * np.transpose(a_old, (0, 2, 1))[..., None]", "o = (o"),
    ("m_new = np.maximum(m, mb)", "m_new = mb"),
    ("return int(np.searchsorted(ks, qp, side=\"right\").sum())", "return int(np.searchsorted(ks, qp, side=\"left\").sum())"),
    ("full += int((vis == total).sum())", "full += int((vis >= total // 2).sum())"),
]


def test_real_ring_oracle_passes_the_pins():
    assert _ring_pins_hold(real_ring)


@pytest.mark.parametrize("find,replace", RING_MUTATIONS)
def test_planted_ring_mistake_is_caught(find, replace):
    assert not _ring_pins_hold(_ring_mutant(find, replace))
