"""ra_ring_forward_noalloc: the entry point for callers that cannot allocate.

Such callers (a latency-critical path where cudaMalloc could synchronise the
device or fail mid-job, or a host framework that owns all device memory) get
ring attention without passing a workspace: the library uses its own fixed
scratch array.  These tests call it through the C ABI and compare it with
ra_ring_forward, and check that oversize problems are refused up front.
This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

import context_exact_attention_ra_gb300 as ra
from workloads import WORKLOADS, make_inputs, small_case


def test_oversize_problem_is_refused_before_anything_runs():
    # s32k needs far more than the 64 MiB scratch: refused with
    # RA_ERR_WORKSPACE, without touching the (null) pointers or a GPU.
    w = WORKLOADS["s32k"]
    shp = ra.Shape(w.B, w.S, w.S, w.Hq, w.Hkv, w.D, ra.BF16, w.scale)
    assert ra.ring_workspace_size(shp, w.c, ra.ZIGZAG, ra.MODE_FUSED) > ra.NOALLOC_SCRATCH_BYTES
    st = ra.lib().ra_ring_forward_noalloc(None, None, None, shp, w.c, ra.ZIGZAG, 1, ra.MODE_FUSED,
                                          ra.BF16, None, None, None)
    assert st == -5
    # argument errors are reported as for ra_ring_forward
    bad = ra.Shape(1, 250, 250, 4, 2, 128, ra.BF16, 0.1)
    assert ra.lib().ra_ring_forward_noalloc(None, None, None, bad, 4, ra.ZIGZAG, 1, 0, ra.BF16,
                                            None, None, None) == -1


@pytest.mark.gpu
def test_noalloc_matches_ring_forward_on_consecutive_calls():
    """Calls in a row, each on fresh inputs (other seeds, layouts and modes,
    so that no call can pass on what the previous one left in the shared
    scratch), each equal bit for bit to ra_ring_forward with a workspace: the
    same kernels run on the same inputs.  The per-step calls keep the
    online-softmax state (o, m, l) in the scratch."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    cases = [
        (WORKLOADS["gqa4k"], "zigzag", "fused"),
        (small_case(2048, 2, "contiguous", True, B=2, Hq=4, Hkv=1, D=128, seed=31), "contiguous", "per_step"),
        (WORKLOADS["gqa4k"].with_(seed=97), "zigzag", "per_step"),
        (small_case(4096, 4, "striped", True, B=1, Hq=8, Hkv=2, D=128, seed=53), "striped", "fused"),
    ]
    stream = torch.cuda.current_stream()
    for w, layout, mode in cases:
        q, k, v, _ = make_inputs(w)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        shp = ra.Shape(w.B, w.S, w.S, w.Hq, w.Hkv, w.D, ra.BF16, w.scale)
        md = ra.MODES[mode]
        assert ra.ring_workspace_size(shp, w.c, ra.LAYOUTS[layout], md) <= ra.NOALLOC_SCRATCH_BYTES
        want, want_lse = ra.ring_forward(qd, kd, vd, w.c, layout, w.causal, mode, scale=w.scale)
        out = torch.full(qd.shape, float("nan"), dtype=qd.dtype, device="cuda")
        lse = torch.full((w.B, w.Hq, w.S), float("nan"), dtype=torch.float32, device="cuda")
        st = ra.lib().ra_ring_forward_noalloc(
            ctypes.c_void_p(qd.data_ptr()), ctypes.c_void_p(kd.data_ptr()), ctypes.c_void_p(vd.data_ptr()),
            shp, w.c, ra.LAYOUTS[layout], int(w.causal), md, ra.BF16,
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
            ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, ra.status_string(st)
        ra.device_error()
        assert torch.equal(out.view(torch.int16), want.view(torch.int16)), (w.name, layout, mode)
        assert torch.equal(lse.view(torch.int32), want_lse.view(torch.int32)), (w.name, layout, mode)
