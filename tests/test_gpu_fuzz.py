"""Randomised GPU parity: shapes drawn from a fixed seed, every path.

Each case draws a sequence length, a rank count, a layout, causal or not,
batch, query and key/value heads and the head dimension, then checks through
the C ABI:
  * the fused ring against the float64 oracle on every row
    ("06 - Sequence / Context Parallelism", section 4 and exercise A: the ring
    result is exact attention);
  * the per-step ring bitwise against the fused one;
  * the all-gather form against the oracle;
  * decode of a few new tokens at random positions over the same keys
    (section 7) against the oracle's definition.
The shapes stay small (S <= 1536) so that the oracle finishes in seconds, but
cover ragged shards, several tiles per shard and every layout.
"""

import numpy as np
import pytest
import torch

import context_exact_attention_ra_gb300 as ra
import oracle
from tests import parity
from workloads import make_inputs, small_case

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


def _draw(i):
    """Case i: a valid shape for its layout (S a multiple of c, of 2c for zig-zag)."""
    r = np.random.RandomState(9000 + i)
    layout = ["contiguous", "zigzag", "striped"][r.randint(3)]
    c = int(r.choice([1, 2, 3, 4, 5, 8]))
    unit = 2 * c if layout == "zigzag" else c
    S = unit * int(r.randint(max(1, 64 // unit), 1536 // unit + 1))
    causal = bool(r.rand() < 0.75)
    Hkv = int(r.choice([1, 2]))
    Hq = Hkv * int(r.choice([1, 2, 4]))
    B = int(r.choice([1, 2]))
    D = int(r.choice([64, 128]))
    return dict(S=S, c=c, layout=layout, causal=causal, B=B, Hq=Hq, Hkv=Hkv, D=D, seed=9100 + i)


CASES = [_draw(i) for i in range(24)]


@pytest.mark.parametrize("case", CASES, ids=[f"{d['layout']}-S{d['S']}-c{d['c']}-D{d['D']}-{'causal' if d['causal'] else 'full'}"
                                             for d in CASES])
def test_random_shapes_every_path(case):
    w = small_case(case["S"], case["c"], case["layout"], case["causal"], B=case["B"], Hq=case["Hq"],
                   Hkv=case["Hkv"], D=case["D"], seed=case["seed"])
    q, k, v, _ = make_inputs(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    pos = np.arange(w.S)
    ref, ref_lse, _, _ = oracle.attention_reference(_np(q), _np(k), _np(v), pos, pos, w.causal, w.scale)

    out, lse = ra.ring_forward(qd, kd, vd, w.c, w.layouts[0], w.causal, "fused", scale=w.scale)
    out_ps, lse_ps = ra.ring_forward(qd, kd, vd, w.c, w.layouts[0], w.causal, "per_step", scale=w.scale)
    out_ag, lse_ag = ra.ring_forward(qd, kd, vd, w.c, w.layouts[0], w.causal, "allgather", scale=w.scale)
    ra.device_error()
    parity.check_bf16(_np(out), ref, "fused out")
    parity.check_lse(_np(lse), ref_lse, "fused lse")
    assert torch.equal(out.view(torch.uint8), out_ps.view(torch.uint8)), "per-step differs from fused"
    assert torch.equal(lse.view(torch.int32), lse_ps.view(torch.int32)), "per-step lse differs from fused"
    parity.check_bf16(_np(out_ag), ref, "all-gather out")
    parity.check_lse(_np(lse_ag), ref_lse, "all-gather lse")

    # decode: R new tokens at random positions against the same keys
    r = np.random.RandomState(case["seed"])
    R = int(r.randint(1, 4))
    q_pos = np.sort(r.choice(w.S, size=R, replace=False)).astype(np.int32)
    qn = torch.randn((w.B, R, w.Hq, w.D), generator=torch.Generator().manual_seed(case["seed"])).to(torch.bfloat16)
    dout, dlse = ra.decode_forward(qn.to(DEV), torch.as_tensor(q_pos, device=DEV), kd, vd, w.c, w.layouts[0],
                                   w.causal, scale=w.scale, out_dtype=torch.float32)
    ra.device_error()
    dref, dref_lse, _, _ = oracle.attention_reference(_np(qn), _np(k), _np(v), q_pos, pos, w.causal, w.scale)
    parity.check_bf16(_np(dout), dref, "decode out")
    assert np.abs(_np(dout) - dref).max() <= 1e-4
    parity.check_lse(_np(dlse), dref_lse, "decode lse")
