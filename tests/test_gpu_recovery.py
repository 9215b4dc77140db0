"""Device-timeout path and resuming a ring from a saved state.

The timeout test runs the library's self-test: one block waits, through the
same bounded wait the attention kernels use, on a barrier nothing arrives on.
The wait must give up, the host must see RA_ERR_TIMEOUT, and the device must
stay usable -- nothing faults or hangs, only the wait runs out.

The resume test stops a rank's ring after step t, copies the online-softmax
state (o, m, l) to the host and back into fresh device buffers, finishes the
ring and checks that the result equals the uninterrupted run bit for bit (the
state after any step is the whole of what the ring carries,
"06 - Sequence / Context Parallelism", section 4).
"""

import numpy as np
import pytest
import torch

import context_exact_attention_ra_gb300 as ra
import oracle
from oracle import ring
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


def test_device_timeout_is_reported_and_the_device_stays_usable():
    assert ra.selftest_wait_timeout(20000) == ra.ERR_TIMEOUT
    ra.device_error()                       # the word was cleared: no error pending
    assert ra.selftest_wait_timeout(1000) == ra.ERR_TIMEOUT
    # ordinary work afterwards
    w = small_case(1024, 2, "zigzag", True, B=1, Hq=4, Hkv=2, D=128, seed=31)
    q, k, v, _ = make_inputs(w)
    out, lse = ra.ring_forward(q.to(DEV), k.to(DEV), v.to(DEV), w.c, "zigzag", True, "fused",
                               scale=w.scale, out_dtype=torch.float32)
    ra.device_error()
    pos = np.arange(w.S)
    ref, ref_lse, _, _ = oracle.attention_reference(_np(q), _np(k), _np(v), pos, pos, True, w.scale)
    parity.check_bf16(_np(out), ref, "after the self-test")
    parity.check_lse(_np(lse), ref_lse, "after the self-test")


def test_pending_device_error_refuses_new_work_until_read():
    """After a wait has run out, and before ra_device_error() has read it,
    every entry point that launches work refuses with RA_ERR_TIMEOUT instead
    of returning RA_OK over stale output; once the error is read and cleared,
    the same calls compute the right result."""
    w = small_case(1024, 2, "zigzag", True, B=1, Hq=4, Hkv=2, D=128, seed=33)
    q, k, v, _ = make_inputs(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    assert ra.selftest_wait_timeout(2000, leave_pending=True) == ra.ERR_TIMEOUT
    sentinel = torch.full(qd.shape, 7.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ra.RaError) as exc:
        ra.ring_forward(qd, kd, vd, w.c, "zigzag", True, "fused", scale=w.scale, out=sentinel)
    assert exc.value.status == ra.ERR_TIMEOUT
    with pytest.raises(ra.RaError) as exc:
        ra.state_init(1, 256, 4, 128)
    assert exc.value.status == ra.ERR_TIMEOUT
    torch.cuda.synchronize()
    assert bool((sentinel == 7.0).all()), "a refused call wrote its output"
    # the pending error is still there for ra_device_error to report, once
    with pytest.raises(ra.RaError) as exc:
        ra.device_error()
    assert exc.value.status == ra.ERR_TIMEOUT
    ra.device_error()
    out, lse = ra.ring_forward(qd, kd, vd, w.c, "zigzag", True, "fused", scale=w.scale,
                               out_dtype=torch.float32)
    ra.device_error()
    pos = np.arange(w.S)
    ref, ref_lse, _, _ = oracle.attention_reference(_np(q), _np(k), _np(v), pos, pos, True, w.scale)
    parity.check_bf16(_np(out), ref, "after the pending error was cleared")
    parity.check_lse(_np(lse), ref_lse, "after the pending error was cleared")


@pytest.mark.parametrize("layout,t_stop", [("zigzag", 1), ("contiguous", 3), ("striped", 2)])
def test_ring_resumes_from_a_saved_state_bit_for_bit(layout, t_stop):
    S, c, rank = 2048, 4, 2
    w = small_case(S, c, layout, True, B=1, Hq=4, Hkv=1, D=128, seed=37)
    q, k, v, _ = make_inputs(w)
    pos = np.asarray(ra.shard_positions(S, c, layout), dtype=np.int32).reshape(c, S // c)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)

    def rows(r):
        idx = torch.as_tensor(pos[r], dtype=torch.long, device=DEV)
        return idx, torch.as_tensor(pos[r], dtype=torch.int32, device=DEV)

    qi_idx, qi_pos = rows(rank)
    qi = qd[:, qi_idx].contiguous()

    def run_steps(o, m, l, steps):
        for t in steps:
            src = ring.ring_source(rank, t, c)
            kj_idx, kj_pos = rows(src)
            ra.block_attn(qi, kd[:, kj_idx].contiguous(), vd[:, kj_idx].contiguous(), qi_pos, kj_pos,
                          True, o, m, l, scale=w.scale)

    # uninterrupted
    o, m, l = ra.state_init(1, S // c, w.Hq, w.D)
    run_steps(o, m, l, range(c))
    out_a, lse_a = ra.lse_merge([o], [m], [l], torch.float32)
    # stopped after t_stop steps, state saved to the host and restored
    o, m, l = ra.state_init(1, S // c, w.Hq, w.D)
    run_steps(o, m, l, range(t_stop))
    torch.cuda.synchronize()
    saved = [x.cpu().clone() for x in (o, m, l)]
    del o, m, l
    o, m, l = (x.to(DEV).contiguous() for x in saved)
    run_steps(o, m, l, range(t_stop, c))
    out_b, lse_b = ra.lse_merge([o], [m], [l], torch.float32)
    ra.device_error()
    assert torch.equal(out_a.view(torch.int32), out_b.view(torch.int32))
    assert torch.equal(lse_a.view(torch.int32), lse_b.view(torch.int32))
    # and the resumed result is this rank's rows of exact attention
    ref, ref_lse, _, _ = oracle.attention_reference(_np(q), _np(k), _np(v), np.arange(S), np.arange(S),
                                                    True, w.scale, rows=pos[rank])
    parity.check_bf16(_np(out_b), ref, "resumed ring")
    parity.check_lse(_np(lse_b), ref_lse, "resumed ring")
