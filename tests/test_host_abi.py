"""The C ABI without a GPU: the library loads, exports every declared entry
point, rejects bad arguments before launching anything, and its host
scheduler agrees bit for bit with the oracle's schedule and work counts."""

import ctypes
import os
import re

import numpy as np
import pytest

import context_exact_attention_ra_gb300 as ra
from oracle import ring

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ra.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ra.LIB_PATH):
        from context_exact_attention_ra_gb300 import _build
        _build.build()
    return ra.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ra_block_attn", "ra_lse_merge", "ra_ring_forward"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    assert ra.status_string(0) == "ok"
    assert "invalid" in ra.status_string(-1)
    assert ra.version().startswith("ra-gb300")


def _shape(B=1, S=256, Hq=4, Hkv=2, D=128, dtype=ra.BF16, scale=0.088):
    return ra.Shape(B, S, S, Hq, Hkv, D, dtype, scale)


@pytest.mark.parametrize("shape,c,layout,code", [
    (_shape(S=250), 4, ra.ZIGZAG, -1),            # S not divisible by 2c
    (_shape(S=250), 3, ra.CONTIGUOUS, -1),        # S not divisible by c
    (_shape(Hq=3, Hkv=2), 2, ra.CONTIGUOUS, -1),  # Hq not a multiple of Hkv
    (_shape(D=96), 2, ra.CONTIGUOUS, -2),         # unsupported head dim
    (_shape(dtype=7), 2, ra.CONTIGUOUS, -2),      # unsupported dtype
    (_shape(scale=0.0), 2, ra.CONTIGUOUS, -1),    # non-positive scale
    (_shape(scale=float("nan")), 2, ra.CONTIGUOUS, -1),
    (_shape(), 0, ra.CONTIGUOUS, -1),             # no ranks
    (_shape(), 2, 5, -1),                         # unknown layout
    (_shape(S=250), 3, ra.STRIPED, -1),           # striped needs S divisible by c
])
def test_ring_forward_rejects_bad_arguments_before_launch(lib, shape, c, layout, code):
    st = lib.ra_ring_forward(None, None, None, shape, c, layout, 1, 0, shape.dtype, None, None, None,
                             0, None, None)
    assert st == code
    assert lib.ra_ring_forward_workspace_size(shape, c, layout, 0) == 0


def test_null_pointers_and_workspace_are_rejected(lib):
    shp = _shape()
    assert lib.ra_ring_forward_workspace_size(shp, 2, ra.ZIGZAG, 0) > 0
    # null inputs
    assert lib.ra_ring_prepare(None, None, None, shp, 2, ra.ZIGZAG, None, 0, None) == -1
    # misaligned inputs
    bad = ctypes.c_void_p(0x1008)
    assert lib.ra_ring_prepare(bad, bad, bad, shp, 2, ra.ZIGZAG, None, 0, None) == -1
    # aligned inputs but no workspace
    ok = ctypes.c_void_p(0x100000)
    assert lib.ra_ring_prepare(ok, ok, ok, shp, 2, ra.ZIGZAG, None, 0, None) == -5
    assert lib.ra_ring_attend(shp, 2, ra.ZIGZAG, 1, 0, ra.BF16, ok, None, ok, 10, 0, None) == -5
    assert lib.ra_ring_attend(shp, 2, ra.ZIGZAG, 1, 9, ra.BF16, ok, None, ok, 10, 0, None) == -1
    # fp32 inputs cannot produce bf16 outputs
    f32 = _shape(dtype=ra.F32)
    assert lib.ra_ring_attend(f32, 2, ra.ZIGZAG, 1, 0, ra.BF16, ok, None, ok, 1 << 30, 0, None) == -1
    assert lib.ra_block_attn(None, None, None, None, None, 1, shp, None, None, None, None, None) == -1
    assert lib.ra_lse_merge(0, None, None, None, shp, None, None, None) == -1
    assert lib.ra_lse_merge(65, None, None, None, shp, None, None, None) == -1


def test_empty_problems_are_noops(lib):
    # B = 0 or S = 0: nothing to do, nothing launched, OK
    assert lib.ra_block_attn(None, None, None, None, None, 1, _shape(B=0), None, None, None, None, None) == 0
    assert lib.ra_ring_forward(None, None, None, _shape(S=0), 2, ra.ZIGZAG, 1, 0, ra.BF16, None, None,
                               None, 0, None, None) == 0
    assert lib.ra_state_init(_shape(S=0), None, None, None, None) == 0


@pytest.mark.parametrize("c", [1, 2, 3, 7, 16])
def test_schedule_matches_oracle(lib, c):
    assert ra.schedule(c) == ring.schedule(c)


@pytest.mark.parametrize("S,c,layout", [(256, 4, "contiguous"), (4096, 4, "zigzag"),
                                        (1000, 5, "zigzag"), (96, 3, "contiguous"),
                                        (96, 3, "striped"), (4096, 16, "striped")])
def test_shard_positions_match_oracle(lib, S, c, layout):
    got = ra.shard_positions(S, c, layout)
    want = np.concatenate(ring.shard_positions(S, c, layout)).tolist()
    assert got == want


@pytest.mark.parametrize("S,c,layout,causal", [
    (256, 4, "contiguous", False), (4096, 4, "zigzag", True), (32768, 8, "contiguous", True),
    (32768, 8, "zigzag", True), (1000, 5, "zigzag", True), (600, 2, "contiguous", True),
    (65536, 8, "zigzag", True), (4096, 4, "striped", True), (1000, 8, "striped", True),
    (32768, 8, "striped", True)])
def test_expected_work_matches_oracle(lib, S, c, layout, causal):
    got = ra.work_expected(S, c, layout, causal)
    want = ring.work_table(S, c, layout, causal)
    for i in range(c):
        for t in range(c):
            assert got[i][t] == (want["pairs"][i, t], want["full"][i, t],
                                 want["partial"][i, t], want["skipped"][i, t]), (i, t)


def test_expected_work_at_c16_reproduces_the_plate():
    S, c = 131072, 16
    got = ra.work_expected(S, c, "contiguous", True)
    per_rank = [sum(got[i][t][0] for t in range(c)) for i in range(c)]
    assert round(max(per_rank) / (sum(per_rank) / c), 2) == 1.94
    z = ra.work_expected(S, c, "zigzag", True)
    zr = [sum(z[i][t][0] for t in range(c)) for i in range(c)]
    assert len(set(zr)) == 1


def test_selftest_rejects_a_bad_limit_before_any_launch(lib):
    assert lib.ra_selftest_wait_timeout(ctypes.c_uint32(0), 0, ctypes.c_void_p(0)) == -1
    assert lib.ra_selftest_wait_timeout(ctypes.c_uint32(2000000), 1, ctypes.c_void_p(0)) == -1


def test_other_entry_points_reject_bad_arguments_before_launch(lib):
    """Host-buffer ring, decode and rotating ring: every argument error is
    caught on the host before any CUDA call (these run without a GPU)."""
    shp = _shape()
    ok = ctypes.c_void_p(0x100000)   # aligned, never dereferenced on these paths
    # host-buffer ring
    hio = lib.ra_ring_forward_hostio
    assert hio(None, None, None, _shape(S=250), 4, ra.ZIGZAG, 1, 0, ra.BF16, None, None, None, 0, None) == -1
    assert hio(None, None, None, shp, 2, ra.ZIGZAG, 1, 9, ra.BF16, None, None, None, 0, None) == -1   # mode
    assert hio(None, None, None, shp, 2, ra.ZIGZAG, 1, 0, 7, None, None, None, 0, None) == -1         # out dtype
    assert hio(None, None, None, shp, 2, ra.ZIGZAG, 1, 0, ra.BF16, None, None, None, 0, None) == -1   # null
    assert hio(ok, ok, ok, shp, 2, ra.ZIGZAG, 1, 0, ra.BF16, ok, None, None, 0, None) == -5           # workspace
    assert hio(None, None, None, _shape(S=0), 2, ra.ZIGZAG, 1, 0, ra.BF16, None, None, None, 0, None) == 0
    assert lib.ra_ring_forward_hostio_workspace_size(_shape(S=250), 4, ra.ZIGZAG, 0, ra.BF16) == 0
    assert (lib.ra_ring_forward_hostio_workspace_size(shp, 2, ra.ZIGZAG, 0, ra.BF16) >
            lib.ra_ring_forward_workspace_size(shp, 2, ra.ZIGZAG, 0))
    # decode: R = 1 new token over S = 256 keys
    dec = lib.ra_decode_forward
    dshp = ra.Shape(1, 1, 256, 4, 2, 128, ra.BF16, 0.088)
    bad_s = ra.Shape(1, 1, 250, 4, 2, 128, ra.BF16, 0.088)
    f32 = ra.Shape(1, 1, 256, 4, 2, 128, ra.F32, 0.088)
    assert dec(None, None, None, None, bad_s, 4, ra.ZIGZAG, 1, ra.BF16, None, None, None, 0, None) == -1
    assert dec(None, None, None, None, f32, 2, ra.ZIGZAG, 1, ra.BF16, None, None, None, 0, None) == -2
    assert dec(None, None, None, None, dshp, 2, ra.ZIGZAG, 1, 7, None, None, None, 0, None) == -1
    assert dec(None, None, None, None, dshp, 2, ra.ZIGZAG, 1, ra.BF16, None, None, None, 0, None) == -1
    assert dec(ok, ok, ok, ok, dshp, 2, ra.ZIGZAG, 1, ra.BF16, ok, None, None, 0, None) == -5
    assert lib.ra_decode_workspace_size(bad_s, 4, ra.ZIGZAG) == 0
    assert lib.ra_decode_workspace_size(dshp, 2, ra.ZIGZAG) > 0
    # rotating ring: overlap needs a copy stream of its own
    rot = lib.ra_ring_forward_rotate
    assert rot(None, None, None, _shape(S=250), 4, ra.ZIGZAG, 1, 0, ra.BF16, None, None, None, 0, None, None) == -1
    assert rot(None, None, None, shp, 2, ra.ZIGZAG, 1, 1, ra.BF16, None, None, None, 0, None, None) == -1
    assert rot(None, None, None, shp, 2, ra.ZIGZAG, 1, 0, ra.BF16, None, None, None, 0, None, None) == -1
    assert rot(ok, ok, ok, shp, 2, ra.ZIGZAG, 1, 0, ra.BF16, ok, None, None, 0, None, None) == -5
