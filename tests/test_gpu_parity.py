"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Every test calls the library (``libra_gb300.so``) through its Python binding
on seeded synthetic inputs and compares with the oracle computed on the CPU
from the same (already rounded) inputs.
"""

import numpy as np
import pytest
import torch

import context_exact_attention_ra_gb300 as ra
import oracle
from oracle import ring
from tests import parity
from workloads import WORKLOADS, make_inputs, small_case

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ra.lib()
    yield
    ra.device_error()


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _run(w, layout, mode="fused", report=False, out_dtype=None):
    q, k, v, offsets = make_inputs(w)
    res = ra.ring_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.c, layout, w.causal, mode,
                          scale=w.scale, report=report, out_dtype=out_dtype)
    ra.device_error()
    return (q, k, v, offsets), res


def _oracle_rows(q, k, v, w, rows):
    pos = np.arange(w.S)
    ref, lse, _, _ = oracle.attention_reference(_np(q), _np(k), _np(v), pos, pos, w.causal,
                                                w.scale, rows=rows)
    return ref, lse


def _oracle_rows_chunked(q, k, v, w, rows, chunk=512):
    """The oracle on `rows`, a few hundred rows per call (bounded host memory)."""
    qn, kn, vn = _np(q), _np(k), _np(v)
    pos = np.arange(w.S)
    refs, lses = [], []
    for a in range(0, len(rows), chunk):
        ref, lse, _, _ = oracle.attention_reference(qn, kn, vn, pos, pos, w.causal, w.scale,
                                                    rows=rows[a:a + chunk])
        refs.append(ref)
        lses.append(lse)
    return np.concatenate(refs, axis=1), np.concatenate(lses, axis=2)


# ---------------------------------------------------------------------------
# Full-size parity on the small workloads
# ---------------------------------------------------------------------------

def test_tiny_fp32_exact_path():
    w = WORKLOADS["tiny"]
    (q, k, v, _), (out, lse) = _run(w, "contiguous")
    ref, ref_lse = _oracle_rows(q, k, v, w, np.arange(w.S))
    parity.check_f32(_np(out), ref, "tiny out")
    fin = np.isfinite(ref_lse)
    rel = np.abs(_np(lse)[fin] - ref_lse[fin]).max() / np.abs(ref_lse[fin]).max()
    assert rel <= parity.F32_REL


def test_gqa4k_full_parity_and_modes_agree_bitwise():
    w = WORKLOADS["gqa4k"]
    (q, k, v, _), (out, lse, info) = _run(w, "zigzag", "fused", report=True)
    ref, ref_lse = _oracle_rows(q, k, v, w, np.arange(w.S))
    parity.check_bf16(_np(out), ref, "gqa4k out")
    parity.check_lse(_np(lse), ref_lse, "gqa4k lse")
    out32, _ = ra.ring_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.c, "zigzag", True, "fused",
                               scale=w.scale, out_dtype=torch.float32)
    parity.check_bf16(_np(out32), ref, "gqa4k out fp32")
    parity.check_rounding(out, out32, "gqa4k")
    out2, lse2 = ra.ring_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.c, "zigzag", True, "per_step",
                                 scale=w.scale)
    out2_32, _ = ra.ring_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.c, "zigzag", True, "per_step",
                                 scale=w.scale, out_dtype=torch.float32)
    ra.device_error()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    assert torch.equal(out32.view(torch.int32), out2_32.view(torch.int32))


@pytest.mark.parametrize("name,layout", [("gqa4k", "zigzag"), ("s32k", "contiguous"),
                                         ("s32k", "zigzag"), ("s32k", "striped"),
                                         ("tiny", "contiguous")])
def test_work_counters_match_host_scheduler_and_oracle(name, layout):
    w = WORKLOADS[name]
    _, (_, _, info) = _run(w, layout, "fused", report=True)
    exp = ra.work_expected(w.S, w.c, layout, w.causal)
    orc = ring.work_table(w.S, w.c, layout, w.causal)
    scale = w.B * w.Hq
    for i in range(w.c):
        for t in range(w.c):
            got = info["per_rank_step"][i][t]
            e = exp[i][t]
            assert (got["pairs"], got["full"], got["partial"], got["skipped"]) == \
                tuple(x * scale for x in e), (i, t)
            assert e == (orc["pairs"][i, t], orc["full"][i, t], orc["partial"][i, t],
                         orc["skipped"][i, t])
    assert info["schedule"] == ring.schedule(w.c)
    per_rank = [sum(info["per_rank_step"][i][t]["pairs"] for t in range(w.c)) for i in range(w.c)]
    if layout == "zigzag":
        assert len(set(per_rank)) == 1
    assert info["ring_kv_bytes"] == ring.ring_kv_bytes(w.S, w.Hkv, w.D, 2 if w.dtype == "bf16" else 4, w.B)


# ---------------------------------------------------------------------------
# Sampled-row parity on the large workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,layout", [("s32k", "contiguous"), ("s32k", "zigzag"),
                                         ("s32k", "striped"), ("s128k", "zigzag"),
                                         ("stress", "zigzag")])
def test_large_workloads_sampled_rows(name, layout):
    w = WORKLOADS[name]
    (q, k, v, offsets), (out32, lse) = _run(w, layout, out_dtype=torch.float32)
    out, lse_b = ra.ring_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.c, layout, w.causal, "fused",
                                 scale=w.scale)
    ra.device_error()
    parity.check_rounding(out, out32, f"{name}/{layout}")
    assert torch.equal(lse.view(torch.int32), lse_b.view(torch.int32))
    # every key row that carries a +50 offset, of every (batch, KV head), is
    # also checked as a query row: it is the first row whose visible set holds
    # that key, and the rows that force the repeated running-max rises
    extra = set()
    for rows in offsets.values():
        extra.update(int(x) for x in rows.tolist())
    rows = parity.sample_rows(w.S, w.c, layout, w.seed, extra=sorted(extra))
    if offsets:
        assert set(rows.tolist()) >= extra
    ref, ref_lse = _oracle_rows_chunked(q, k, v, w, rows)
    got = _np(out32[:, torch.as_tensor(rows)])
    parity.check_bf16(got, ref, f"{name}/{layout} out")
    parity.check_lse(_np(lse[:, :, torch.as_tensor(rows)]), ref_lse, f"{name}/{layout} lse",
                     report=True)
    # properties that hold for every row: finite, and |out| bounded by max |v|
    o = out32
    assert torch.isfinite(o).all()
    assert o.abs().max().item() <= v.float().abs().max().item() * (1 + 1e-2) + 1e-2
    assert torch.isfinite(lse).all()


# ---------------------------------------------------------------------------
# Edge cases: ragged shards, D=64, batch > 1, c = 1, tiny chunks
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S,c,layout,causal,B,Hq,Hkv,D,dtype", [
    (1000, 5, "zigzag", True, 1, 4, 2, 128, "bf16"),        # chunks of 100 rows
    (600, 2, "contiguous", False, 2, 2, 1, 128, "bf16"),    # shards of 300 rows
    (768, 3, "contiguous", True, 1, 4, 4, 64, "bf16"),      # D = 64, MHA
    (512, 1, "contiguous", True, 2, 8, 1, 128, "bf16"),     # one rank
    (256, 64, "zigzag", True, 1, 2, 1, 128, "bf16"),        # chunks of 2 rows
    (384, 3, "zigzag", True, 1, 2, 1, 128, "f32"),          # fp32, D = 128, ragged tiles
    (200, 4, "contiguous", True, 2, 4, 2, 64, "f32"),
    (1024, 4, "striped", True, 1, 4, 2, 128, "bf16"),       # round-robin tokens
    (1000, 8, "striped", True, 2, 2, 1, 64, "bf16"),        # ragged striped shards
    (384, 3, "striped", True, 1, 2, 1, 128, "f32"),
])
def test_edge_cases_full_parity(S, c, layout, causal, B, Hq, Hkv, D, dtype):
    w = small_case(S, c, layout, causal, B=B, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, seed=S + c)
    (q, k, v, _), (out, lse, info) = _run(w, layout, "fused", report=True)
    ref, ref_lse = _oracle_rows(q, k, v, w, np.arange(S))
    if dtype == "bf16":
        parity.check_bf16(_np(out), ref, "edge out")
        parity.check_lse(_np(lse), ref_lse, "edge lse")
    else:
        parity.check_f32(_np(out), ref, "edge out")
    out2, lse2 = ra.ring_forward(q.to(DEV), k.to(DEV), v.to(DEV), c, layout, causal, "per_step",
                                 scale=w.scale)
    ra.device_error()
    assert torch.equal(out.view(torch.uint8), out2.view(torch.uint8))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    exp = ra.work_expected(S, c, layout, causal)
    for i in range(c):
        for t in range(c):
            got = info["per_rank_step"][i][t]
            assert (got["pairs"], got["full"], got["partial"], got["skipped"]) == \
                tuple(x * B * Hq for x in exp[i][t])


def test_empty_sequence_is_a_noop():
    q = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device=DEV)
    k = torch.empty((1, 0, 1, 128), dtype=torch.bfloat16, device=DEV)
    out, lse = ra.ring_forward(q, k, k, 2, "zigzag", True, "fused", workspace=torch.empty(256, dtype=torch.uint8, device=DEV))
    assert out.numel() == 0 and lse.numel() == 0


# ---------------------------------------------------------------------------
# ra_block_attn and ra_lse_merge on their own
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_block_attn_arbitrary_positions_and_state(dtype):
    # one rank's queries against two held blocks, positions scrambled
    rng = np.random.default_rng(3)
    B, Sq, Sk, Hq, Hkv, D = 2, 300, 260, 4, 2, 128
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(7)
    q = torch.randn((B, Sq, Hq, D), generator=g).to(tdt)
    k1 = torch.randn((B, Sk, Hkv, D), generator=g).to(tdt)
    v1 = torch.randn((B, Sk, Hkv, D), generator=g).to(tdt)
    k2 = torch.randn((B, Sk, Hkv, D), generator=g).to(tdt)
    v2 = torch.randn((B, Sk, Hkv, D), generator=g).to(tdt)
    perm = rng.permutation(2000)
    qp, kp1, kp2 = perm[:Sq], perm[Sq:Sq + Sk], perm[Sq + Sk:Sq + 2 * Sk]
    scale = D ** -0.5
    o, m, l = ra.state_init(B, Sq, Hq, D)
    work = torch.zeros(4, dtype=torch.int64, device=DEV)
    for kk, vv, kp in ((k1, v1, kp1), (k2, v2, kp2)):
        ra.block_attn(q.to(DEV), kk.to(DEV), vv.to(DEV), torch.as_tensor(qp, dtype=torch.int32, device=DEV),
                      torch.as_tensor(kp, dtype=torch.int32, device=DEV), True, o, m, l, scale=scale,
                      work=work)
    ra.device_error()
    # the state after both blocks: compare with the oracle's partial over the union
    K = torch.cat([k1, k2], 1)
    V = torch.cat([v1, v2], 1)
    kp = np.concatenate([kp1, kp2])
    ob, mb, lb = ring.block_partial(_np(q), _np(K), _np(V), qp, kp, True, scale)
    m_nat = _np(m) * np.log(2.0)
    fin = np.isfinite(mb)
    assert (np.isfinite(m_nat) == fin).all()
    # state normalised by its own l equals the oracle's normalised output
    out = _np(o) / np.where(_np(l) > 0, _np(l), 1.0).transpose(0, 2, 1)[..., None]
    ref = ob / np.where(lb > 0, lb, 1.0).transpose(0, 2, 1)[..., None]
    lse = np.where(_np(l) > 0, m_nat + np.log(np.where(_np(l) > 0, _np(l), 1.0)), -np.inf)
    ref_lse = np.where(lb > 0, mb + np.log(np.where(lb > 0, lb, 1.0)), -np.inf)
    if dtype == "bf16":
        parity.check_bf16(out, ref, "block out")
    else:
        parity.check_f32(out, ref, "block out")
    parity.check_lse(lse, ref_lse, "block lse")
    pairs = ring.visible_pairs(qp, kp1, True) + ring.visible_pairs(qp, kp2, True)
    assert int(work[0].item()) == pairs * B * Hq


# P = 2-4 take the all-loads-first merge, P = 9 and 64 the general merge
# through more than one pass of per-partial weights (eight partials per pass);
# D = 64 the two-column-per-lane forms
@pytest.mark.parametrize("P,D", [(1, 128), (2, 128), (3, 128), (4, 128), (9, 128), (64, 128), (2, 64), (9, 64)])
def test_lse_merge_of_key_splits_equals_full_attention(P, D):
    B, S, Hq, Hkv = 1, 512, 4, 1
    g = torch.Generator().manual_seed(11)
    q = torch.randn((B, S, Hq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((B, S, Hkv, D), generator=g).to(torch.bfloat16)
    v = torch.randn((B, S, Hkv, D), generator=g).to(torch.bfloat16)
    pos = torch.arange(S, dtype=torch.int32, device=DEV)
    edges = np.linspace(0, S, P + 1).astype(int)
    outs, ms, ls = [], [], []
    for a, b in zip(edges[:-1], edges[1:]):
        o, m, l = ra.state_init(B, S, Hq, D)
        ra.block_attn(q.to(DEV), k[:, a:b].contiguous().to(DEV), v[:, a:b].contiguous().to(DEV),
                      pos, pos[a:b].contiguous(), True, o, m, l)
        outs.append(o)
        ms.append(m)
        ls.append(l)
    out, lse = ra.lse_merge(outs, ms, ls, torch.bfloat16)
    out32, _ = ra.lse_merge(outs, ms, ls, torch.float32)
    ra.device_error()
    ref, ref_lse, _, _ = oracle.attention_reference(_np(q), _np(k), _np(v), np.arange(S), np.arange(S),
                                                    True, D ** -0.5)
    parity.check_bf16(_np(out), ref, "merge out")
    parity.check_bf16(_np(out32), ref, "merge out f32")
    parity.check_lse(_np(lse), ref_lse, "merge lse")


# Pinned outputs are written by the kernels directly, pageable ones are copied.
# The fused ring with pinned queries and outputs in the contiguous or zig-zag
# layout runs pipelined (K and V packed first, each rank's query rows copied and
# its blocks launched on their own); the other cases go through one launch.
@pytest.mark.parametrize("mode,pinned_out,layout,B,pinned_kv,out_f32,S,c", [
    ("fused", True, "zigzag", 1, True, False, 2048, 4),
    ("fused", False, "zigzag", 1, True, False, 2048, 4),
    ("per_step", True, "zigzag", 1, True, False, 2048, 4),
    ("fused", True, "contiguous", 2, True, False, 2048, 4),
    ("fused", True, "zigzag", 2, False, False, 2048, 4),
    ("fused", True, "striped", 1, True, False, 2048, 4),
    ("fused", True, "zigzag", 1, True, True, 2048, 4),
    ("fused", True, "zigzag", 1, True, False, 4096, 16),   # 16 launches of one block row each
])
def test_hostio_equals_device_path(mode, pinned_out, layout, B, pinned_kv, out_f32, S, c):
    w = small_case(S, c, layout, True, B=B, Hq=4, Hkv=1, D=128, seed=21)
    q, k, v, _ = make_inputs(w)
    odt = torch.float32 if out_f32 else None
    out_d, lse_d = ra.ring_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.c, layout, True, mode, out_dtype=odt)
    qh = q.pin_memory()
    kh, vh = (k.pin_memory(), v.pin_memory()) if pinned_kv else (k.clone(), v.clone())
    out_h = torch.empty(q.shape, dtype=torch.float32) if out_f32 else torch.empty_like(qh)
    lse_h = torch.empty((B, w.Hq, w.S), dtype=torch.float32)
    if pinned_out:
        out_h, lse_h = out_h.pin_memory(), lse_h.pin_memory()
    bits = torch.int32 if out_f32 else torch.int16
    for _ in range(2):   # the second call reuses the internal streams and events
        ra.ring_forward_hostio(qh, kh, vh, w.c, layout, True, mode, out_host=out_h, lse_host=lse_h)
        assert torch.equal(out_h.view(bits), out_d.cpu().view(bits))
        assert torch.equal(lse_h.view(torch.int32), lse_d.cpu().view(torch.int32))


def test_hostio_concurrent_threads_on_one_device():
    """Two host threads call the pipelined host-buffer ring on one device at
    once, with different c (the second needs more events than any call before
    it, so the shared event pool grows while the other thread runs), each with
    its own stream and workspace: both results equal the device path bit for
    bit on every call."""
    import threading

    cases = [small_case(2048, 4, "zigzag", True, B=1, Hq=4, Hkv=1, D=128, seed=61),
             small_case(8192, 32, "zigzag", True, B=1, Hq=2, Hkv=1, D=128, seed=62)]
    prepared = []
    for w in cases:
        q, k, v, _ = make_inputs(w)
        want, want_lse = ra.ring_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.c, "zigzag", True, "fused",
                                         scale=w.scale)
        qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
        oh = torch.empty_like(qh).pin_memory()
        lh = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32).pin_memory()
        shp = ra.Shape(w.B, w.S, w.S, w.Hq, w.Hkv, w.D, ra.BF16, w.scale)
        ws = torch.empty(ra.hostio_workspace_size(shp, w.c, ra.ZIGZAG, ra.MODE_FUSED),
                         dtype=torch.uint8, device=DEV)
        prepared.append((w, qh, kh, vh, oh, lh, ws, torch.cuda.Stream(), want.cpu(), want_lse.cpu()))
    torch.cuda.synchronize()
    start = threading.Barrier(len(prepared))
    errors = []

    def worker(w, qh, kh, vh, oh, lh, ws, st, want, want_lse):
        try:
            start.wait()
            for _ in range(3):
                ra.ring_forward_hostio(qh, kh, vh, w.c, "zigzag", True, "fused", w.scale, oh, lh, ws,
                                       stream=st)
                if not torch.equal(oh.view(torch.int16), want.view(torch.int16)) or \
                        not torch.equal(lh.view(torch.int32), want_lse.view(torch.int32)):
                    errors.append(f"{w.name}: result differs from the device path")
        except Exception as e:  # reported below, in the test's thread
            errors.append(f"{w.name}: {e!r}")

    threads = [threading.Thread(target=worker, args=a) for a in prepared]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads)
    ra.device_error()
    assert not errors, errors


# ---------------------------------------------------------------------------
# The all-gather form (one step over the gathered keys) and striped shards
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,layout", [("gqa4k", "zigzag"), ("tiny", "contiguous"),
                                         ("gqa4k", "striped")])
def test_allgather_mode_full_parity_and_counters(name, layout):
    w = WORKLOADS[name]
    q, k, v, _ = make_inputs(w)
    out, lse, info = ra.ring_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.c, layout, w.causal,
                                     "allgather", scale=w.scale, report=True)
    ra.device_error()
    ref, ref_lse = _oracle_rows(q, k, v, w, np.arange(w.S))
    if w.dtype == "bf16":
        parity.check_bf16(_np(out), ref, "allgather out")
        parity.check_lse(_np(lse), ref_lse, "allgather lse")
    else:
        parity.check_f32(_np(out), ref, "allgather out")
    # counters: rank i against the gathered keys, all at step 0
    shards = ring.shard_positions(w.S, w.c, layout)
    gathered = np.concatenate(shards)
    for i in range(w.c):
        got = info["per_rank_step"][i][0]
        f, p_, s_ = ring.tile_classes(shards[i], gathered, w.causal)
        pairs = ring.visible_pairs(shards[i], gathered, w.causal)
        scale = w.B * w.Hq
        assert (got["pairs"], got["full"], got["partial"], got["skipped"]) == \
            (pairs * scale, f * scale, p_ * scale, s_ * scale)
        assert all(info["per_rank_step"][i][t]["pairs"] == 0 for t in range(1, w.c))


def test_allgather_large_sampled_rows():
    w = WORKLOADS["s32k"]
    q, k, v, _ = make_inputs(w)
    out, lse = ra.ring_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.c, "zigzag", True, "allgather",
                               scale=w.scale, out_dtype=torch.float32)
    ra.device_error()
    rows = parity.sample_rows(w.S, w.c, "zigzag", w.seed)
    ref, ref_lse = _oracle_rows(q, k, v, w, rows)
    parity.check_bf16(_np(out[:, torch.as_tensor(rows)]), ref, "allgather s32k out")
    parity.check_lse(_np(lse[:, :, torch.as_tensor(rows)]), ref_lse, "allgather s32k lse")


# ---------------------------------------------------------------------------
# Decode over distributed keys: split-K partials per shard piece + merge
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S,c,layout,R,Hq,Hkv,D,B", [
    (4096, 4, "zigzag", 1, 8, 2, 128, 1),        # one new token, GQA 4:1
    (4096, 4, "contiguous", 4, 8, 2, 128, 2),    # a few tokens at mixed positions, batch 2
    (3000, 5, "striped", 3, 6, 3, 64, 1),        # ragged last tile, D = 64
    (3000, 5, "striped", 3, 6, 3, 128, 1),       # striped shards on the tensor cores, ragged last tile
    (8192, 4, "striped", 1, 16, 1, 128, 2),      # striped, every tile full, batch 2
    (3000, 5, "zigzag", 3, 6, 3, 128, 1),        # zig-zag chunks of 300 keys: two ragged tiles per shard
    (6200, 4, "zigzag", 2, 8, 1, 128, 2),        # chunks of 775 keys, batch 2
    (2600, 4, "contiguous", 2, 8, 2, 64, 1),     # D = 64, contiguous
    (2400, 4, "zigzag", 1, 16, 1, 64, 2),        # D = 64, zig-zag chunks of 300 keys, batch 2
    (2048, 4, "zigzag", 4, 64, 8, 128, 4),       # 64 (batch, head, row block) units, 3 partials each
    (131072, 16, "zigzag", 1, 16, 1, 128, 1),    # the s128k shape: 16 query heads share one KV head
    (131072, 16, "striped", 1, 16, 1, 128, 1),   # the same keys in striped shards (strided tensor map)
])
def test_decode_split_kv_full_parity(S, c, layout, R, Hq, Hkv, D, B):
    g = torch.Generator().manual_seed(S + R)
    k = torch.randn((B, S, Hkv, D), generator=g).to(torch.bfloat16)
    v = torch.randn((B, S, Hkv, D), generator=g).to(torch.bfloat16)
    q = torch.randn((B, R, Hq, D), generator=g).to(torch.bfloat16)
    q_pos = np.array(sorted({S - 1, S // 2, 17, S // 3}))[:R] if R > 1 else np.array([S - 1])
    q_pos = q_pos[:R]
    out, lse = ra.decode_forward(q.to(DEV), torch.as_tensor(q_pos, dtype=torch.int32, device=DEV),
                                 k.to(DEV), v.to(DEV), c, layout, True, out_dtype=torch.float32)
    outb, _ = ra.decode_forward(q.to(DEV), torch.as_tensor(q_pos, dtype=torch.int32, device=DEV),
                                k.to(DEV), v.to(DEV), c, layout, True)
    ra.device_error()
    scale = D ** -0.5
    ref, ref_lse, _ = ring.decode_split_kv(_np(q), q_pos, _np(k), _np(v), c, layout, True, scale)
    ref2, ref2_lse, _, _ = oracle.attention_reference(_np(q), _np(k), _np(v), q_pos, np.arange(S), True, scale)
    assert np.allclose(ref, ref2, atol=1e-10)
    # fp32 arithmetic throughout: the result is close to the float64 oracle
    parity.check_bf16(_np(out), ref, "decode out")
    assert np.abs(_np(out) - ref).max() <= 1e-4
    parity.check_lse(_np(lse), ref_lse, "decode lse")
    parity.check_rounding(outb, out, "decode")


# ---------------------------------------------------------------------------
# The ring with its K/V pass made real (device-to-device rotation), with and
# without overlap: bitwise equal to the per-step mode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,layout,overlap", [("gqa4k", "zigzag", True), ("gqa4k", "zigzag", False),
                                                 ("tiny", "contiguous", True), ("gqa4k", "striped", True)])
def test_rotating_ring_equals_per_step(name, layout, overlap):
    w = WORKLOADS[name]
    q, k, v, _ = make_inputs(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    want, want_lse = ra.ring_forward(qd, kd, vd, w.c, layout, w.causal, "per_step", scale=w.scale)
    got, got_lse = ra.ring_forward_rotate(qd, kd, vd, w.c, layout, w.causal, overlap, scale=w.scale)
    torch.cuda.synchronize()
    ra.device_error()
    assert torch.equal(got.view(torch.uint8), want.view(torch.uint8))
    assert torch.equal(got_lse.view(torch.int32), want_lse.view(torch.int32))


def test_rotating_ring_ragged_batch():
    w = small_case(1000, 5, "zigzag", True, B=2, Hq=4, Hkv=2, D=128, seed=41)
    q, k, v, _ = make_inputs(w)
    got, _ = ra.ring_forward_rotate(q.to(DEV), k.to(DEV), v.to(DEV), w.c, "zigzag", True, True)
    torch.cuda.synchronize()
    ra.device_error()
    ref, _ = _oracle_rows(q, k, v, w, np.arange(w.S))
    parity.check_bf16(_np(got), ref, "rotating ring out")
