"""ra_ring_forward_noalloc: the entry point for callers that cannot allocate.

Such callers (a latency-critical path where cudaMalloc could synchronise the
device or fail mid-job, or a host framework that owns all device memory) get
ring attention without passing a workspace: the library uses its own fixed
scratch array.  These tests call it through the C ABI and compare it with
ra_ring_forward, and check that oversize problems are refused up front.
This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import context_exact_attention_ra_gb300 as ra
from tests import parity
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
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    cases = [(WORKLOADS["gqa4k"], "zigzag"),
             (small_case(2048, 2, "contiguous", True, B=2, Hq=4, Hkv=1, D=128, seed=31), "contiguous"),
             (WORKLOADS["gqa4k"], "zigzag")]
    for w, layout in cases:
        q, k, v, _ = make_inputs(w)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        shp = ra.Shape(w.B, w.S, w.S, w.Hq, w.Hkv, w.D, ra.BF16, w.scale)
        assert ra.ring_workspace_size(shp, w.c, ra.LAYOUTS[layout], ra.MODE_FUSED) <= ra.NOALLOC_SCRATCH_BYTES
        want, want_lse = ra.ring_forward(qd, kd, vd, w.c, layout, w.causal, "fused", scale=w.scale)
        out = torch.empty_like(qd)
        lse = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device="cuda")
        st = ra.lib().ra_ring_forward_noalloc(
            ctypes.c_void_p(qd.data_ptr()), ctypes.c_void_p(kd.data_ptr()), ctypes.c_void_p(vd.data_ptr()),
            shp, w.c, ra.LAYOUTS[layout], int(w.causal), ra.MODE_FUSED, ra.BF16,
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0
        ra.device_error()
        parity.check_bf16(out.double().cpu().numpy(), want.double().cpu().numpy(), "noalloc out")
        parity.check_lse(lse.double().cpu().numpy(), want_lse.double().cpu().numpy(), "noalloc lse")
        assert np.isfinite(out.float().cpu().numpy()).all()
