"""Exact ring attention on GB300 (sm_103a): Python binding of ``libra_gb300.so``.

Argument marshalling only: tensors are passed to the C ABI (``include/ra.h``)
as raw device pointers with the current CUDA stream, and every step of the
computation runs in the library's kernels.  PyTorch supplies device memory
and streams.  If the library is missing, every call raises; there is no
fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "RaError", "lib", "Shape", "Work", "Report", "BF16", "F32", "CONTIGUOUS", "ZIGZAG",
    "MODE_FUSED", "MODE_PER_STEP", "ring_forward", "ring_forward_hostio", "ring_prepare",
    "ring_attend", "ring_read_work", "ring_workspace_size", "block_attn", "state_init",
    "lse_merge", "schedule", "shard_positions", "work_expected", "device_error", "version",
    "LAYOUTS", "MODES",
]

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libra_gb300.so")

BF16, F32 = 0, 1
CONTIGUOUS, ZIGZAG, STRIPED = 0, 1, 2
MODE_FUSED, MODE_PER_STEP, MODE_ALLGATHER = 0, 1, 2
LAYOUTS = {"contiguous": CONTIGUOUS, "zigzag": ZIGZAG, "striped": STRIPED}
MODES = {"fused": MODE_FUSED, "per_step": MODE_PER_STEP, "allgather": MODE_ALLGATHER}
MERGE_MAX_PARTIALS = 64
OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = 0, -1, -2, -3, -4, -5


class RaError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        detail = ""
        try:
            detail = lib().ra_last_error().decode()
        except Exception:  # library not loadable
            pass
        msg = f"{what}: {status_string(status)} ({status})"
        super().__init__(f"{msg} [{detail}]" if detail and status in (-3, -4) else msg)


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Sq", ctypes.c_int32), ("Sk", ctypes.c_int32),
                ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float)]


class Work(ctypes.Structure):
    _fields_ = [("pairs", ctypes.c_uint64), ("tiles_full", ctypes.c_uint64),
                ("tiles_partial", ctypes.c_uint64), ("tiles_skipped", ctypes.c_uint64)]


class Report(ctypes.Structure):
    _fields_ = [("c", ctypes.c_int32), ("per_rank_step", ctypes.POINTER(Work)),
                ("schedule", ctypes.POINTER(ctypes.c_int32)),
                ("imbalance_pairs", ctypes.c_double), ("imbalance_tiles", ctypes.c_double),
                ("ring_kv_bytes", ctypes.c_uint64), ("ring_kv_bytes_sent", ctypes.c_uint64),
                ("algorithmic_flop", ctypes.c_uint64)]


_P = ctypes.c_void_p
_SIGS = {
    "ra_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ra_version": (ctypes.c_char_p, []),
    "ra_last_error": (ctypes.c_char_p, []),
    "ra_state_init": (ctypes.c_int, [Shape, _P, _P, _P, _P]),
    "ra_block_attn": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int, Shape, _P, _P, _P, _P, _P]),
    "ra_lse_merge": (ctypes.c_int, [ctypes.c_int, _P, _P, _P, Shape, _P, _P, _P]),
    "ra_ring_forward_workspace_size": (ctypes.c_size_t, [Shape, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "ra_ring_forward": (ctypes.c_int, [_P, _P, _P, Shape, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, _P, _P, _P, ctypes.c_size_t,
                                       ctypes.POINTER(Report), _P]),
    "ra_ring_prepare": (ctypes.c_int, [_P, _P, _P, Shape, ctypes.c_int, ctypes.c_int, _P,
                                       ctypes.c_size_t, _P]),
    "ra_ring_attend": (ctypes.c_int, [Shape, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, _P, _P, _P, ctypes.c_size_t, ctypes.c_int, _P]),
    "ra_ring_read_work": (ctypes.c_int, [Shape, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P,
                                         ctypes.c_size_t, ctypes.POINTER(Work), _P]),
    "ra_ring_forward_hostio_workspace_size": (ctypes.c_size_t, [Shape, ctypes.c_int, ctypes.c_int,
                                                                ctypes.c_int, ctypes.c_int]),
    "ra_ring_forward_hostio": (ctypes.c_int, [_P, _P, _P, Shape, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P,
                                              ctypes.c_size_t, _P]),
    "ra_ring_rotate_workspace_size": (ctypes.c_size_t, [Shape, ctypes.c_int, ctypes.c_int]),
    "ra_ring_forward_rotate": (ctypes.c_int, [_P, _P, _P, Shape, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, _P, _P, _P, ctypes.c_size_t,
                                              _P, _P]),
    "ra_decode_workspace_size": (ctypes.c_size_t, [Shape, ctypes.c_int, ctypes.c_int]),
    "ra_decode_forward": (ctypes.c_int, [_P, _P, _P, _P, Shape, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, _P, _P, _P, ctypes.c_size_t, _P]),
    "ra_schedule": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_int32)]),
    "ra_shard_positions": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(ctypes.c_int32)]),
    "ra_work_expected": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(Work)]),
    "ra_device_error": (ctypes.c_int, [_P]),
    "ra_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, ctypes.c_int, _P]),
    "ra_ring_forward_noalloc": (ctypes.c_int, [_P, _P, _P, Shape, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P]),
}

_lib = None


def lib():
    """The loaded library (loaded on first use; raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status):
    try:
        return lib().ra_status_string(int(status)).decode()
    except Exception:  # library not loadable
        return "status"


def version():
    return lib().ra_version().decode()


def _check(status, what):
    if status != 0:
        raise RaError(status, what)


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _shape(q, k, scale):
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    return Shape(B, Sq, Sk, Hq, Hkv, D, _dtype_code(q), float(scale))


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def ring_workspace_size(shape: Shape, c, layout, mode):
    return int(lib().ra_ring_forward_workspace_size(shape, int(c), int(layout), int(mode)))


def _out_code(out_dtype, q):
    dt = q.dtype if out_dtype is None else out_dtype
    return _dtype_code(torch.empty(0, dtype=dt)), dt


def ring_forward(q, k, v, c, layout="zigzag", causal=True, mode="fused", scale=None,
                 workspace=None, report=False, stream=None, out_dtype=None, out=None, lse=None):
    """Ring attention of q [B,S,Hq,D] over k, v [B,S,Hkv,D] with c virtual ranks.

    Returns (out [B,S,Hq,D] in out_dtype (default q's dtype; torch.float32
    gives the result before its rounding to bf16), lse [B,Hq,S] float32) and,
    with ``report=True``, a dict of per-(rank, step) work counted on the GPU,
    the ring schedule and the derived quantities.  ``out`` and ``lse`` may be
    given (contiguous, of those shapes; out's dtype then sets out_dtype).
    """
    _contig(q, k, v)
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    md = MODES[mode] if isinstance(mode, str) else int(mode)
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    shp = _shape(q, k, scale)
    ocode, odt = _out_code(out.dtype if out is not None else out_dtype, q)
    if out is None:
        out = torch.empty(q.shape, dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=q.device)
    _contig(out, lse)
    need = ring_workspace_size(shp, c, lay, md)
    if need == 0 and q.numel() > 0:
        raise RaError(-1, "ra_ring_forward_workspace_size")
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rep = None
    work = None
    sched = None
    if report:
        work = (Work * (c * c))()
        sched = (ctypes.c_int32 * (c * c))()
        rep = Report(c, ctypes.cast(work, ctypes.POINTER(Work)),
                     ctypes.cast(sched, ctypes.POINTER(ctypes.c_int32)), 0, 0, 0, 0, 0)
    st = lib().ra_ring_forward(_ptr(q), _ptr(k), _ptr(v), shp, int(c), lay, int(bool(causal)), md,
                               ocode, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                               ctypes.byref(rep) if rep is not None else None, _stream(stream))
    _check(st, "ra_ring_forward")
    if not report:
        return out, lse
    info = {
        "per_rank_step": [[dict(pairs=work[i * c + t].pairs, full=work[i * c + t].tiles_full,
                                partial=work[i * c + t].tiles_partial,
                                skipped=work[i * c + t].tiles_skipped) for t in range(c)]
                          for i in range(c)],
        "schedule": [[sched[t * c + i] for i in range(c)] for t in range(c)],
        "imbalance_pairs": rep.imbalance_pairs,
        "imbalance_tiles": rep.imbalance_tiles,
        "ring_kv_bytes": rep.ring_kv_bytes,
        "ring_kv_bytes_sent": rep.ring_kv_bytes_sent,
        "algorithmic_flop": rep.algorithmic_flop,
    }
    return out, lse, info


def ring_prepare(q, k, v, c, layout, workspace, scale=None, stream=None):
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    st = lib().ra_ring_prepare(_ptr(q), _ptr(k), _ptr(v), _shape(q, k, scale), int(c), lay,
                               _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "ra_ring_prepare")


def ring_attend(shape: Shape, c, layout, causal, mode, out, lse, workspace, count_work=False,
                stream=None):
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    md = MODES[mode] if isinstance(mode, str) else int(mode)
    st = lib().ra_ring_attend(shape, int(c), lay, int(bool(causal)), md, _dtype_code(out),
                              _ptr(out), _ptr(lse),
                              _ptr(workspace), workspace.numel(), int(bool(count_work)),
                              _stream(stream))
    _check(st, "ra_ring_attend")


def ring_read_work(shape: Shape, c, layout, mode, workspace, stream=None):
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    md = MODES[mode] if isinstance(mode, str) else int(mode)
    work = (Work * (c * c))()
    st = lib().ra_ring_read_work(shape, int(c), lay, md, _ptr(workspace), workspace.numel(),
                                 work, _stream(stream))
    _check(st, "ra_ring_read_work")
    return [[(work[i * c + t].pairs, work[i * c + t].tiles_full, work[i * c + t].tiles_partial,
              work[i * c + t].tiles_skipped) for t in range(c)] for i in range(c)]


def ring_forward_hostio(q_host, k_host, v_host, c, layout="zigzag", causal=True, mode="fused",
                        scale=None, out_host=None, lse_host=None, workspace=None, stream=None):
    """ring_forward with host (ideally pinned) CPU tensors in and out; the
    library copies the inputs to the device inside the call, and the kernels
    write pinned outputs directly (pageable outputs are copied back)."""
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    md = MODES[mode] if isinstance(mode, str) else int(mode)
    scale = q_host.shape[-1] ** -0.5 if scale is None else scale
    shp = _shape(q_host, k_host, scale)
    if out_host is None:
        out_host = torch.empty_like(q_host)
    ocode = _dtype_code(out_host)
    need = int(lib().ra_ring_forward_hostio_workspace_size(shp, int(c), lay, md, ocode))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    st = lib().ra_ring_forward_hostio(_ptr(q_host), _ptr(k_host), _ptr(v_host), shp, int(c), lay,
                                      int(bool(causal)), md, ocode, _ptr(out_host), _ptr(lse_host),
                                      _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "ra_ring_forward_hostio")
    return out_host, lse_host


def hostio_workspace_size(shape: Shape, c, layout, mode, out_dtype_code=None):
    oc = shape.dtype if out_dtype_code is None else out_dtype_code
    return int(lib().ra_ring_forward_hostio_workspace_size(shape, int(c), int(layout), int(mode), oc))


def ring_forward_rotate(q, k, v, c, layout="zigzag", causal=True, overlap=True, scale=None,
                        out_dtype=None, workspace=None, stream=None, copy_stream=None):
    """The ring with real K/V rotation between steps (device-to-device
    copies), overlapped with the attention on ``copy_stream`` or not."""
    _contig(q, k, v)
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    shp = _shape(q, k, scale)
    ocode, odt = _out_code(out_dtype, q)
    out = torch.empty(q.shape, dtype=odt, device=q.device)
    lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = int(lib().ra_ring_rotate_workspace_size(shp, int(c), lay))
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if overlap and copy_stream is None:
        copy_stream = torch.cuda.Stream(device=q.device)
    cs = ctypes.c_void_p(copy_stream.cuda_stream) if (overlap and copy_stream is not None) else ctypes.c_void_p(0)
    st = lib().ra_ring_forward_rotate(_ptr(q), _ptr(k), _ptr(v), shp, int(c), lay, int(bool(causal)),
                                      int(bool(overlap)), ocode, _ptr(out), _ptr(lse), _ptr(workspace),
                                      workspace.numel(), _stream(stream), cs)
    _check(st, "ra_ring_forward_rotate")
    return out, lse


def decode_forward(q, q_pos, k, v, c, layout="zigzag", causal=True, scale=None, out_dtype=None,
                   workspace=None, stream=None, out=None, lse=None):
    """Attention of a few new tokens' queries q [B,R,Hq,D] (positions q_pos,
    int32 [R]) over k, v [B,S,Hkv,D] held in c shards: split-K partials per
    shard piece, then their merge.  Returns (out [B,R,Hq,D], lse [B,Hq,R]);
    ``out``, ``lse`` and ``workspace`` may be given to reuse buffers."""
    _contig(q, k, v)
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    B, R, Hq, D = q.shape
    shp = Shape(B, R, k.shape[1], Hq, k.shape[2], D, _dtype_code(q), float(scale))
    ocode, odt = _out_code(out_dtype, q)
    if out is None:
        out = torch.empty((B, R, Hq, D), dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, R), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = int(lib().ra_decode_workspace_size(shp, int(c), lay))
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().ra_decode_forward(_ptr(q), _ptr(q_pos), _ptr(k), _ptr(v), shp, int(c), lay,
                                 int(bool(causal)), ocode, _ptr(out), _ptr(lse), _ptr(workspace),
                                 workspace.numel(), _stream(stream))
    _check(st, "ra_decode_forward")
    return out, lse


def state_init(B, S, Hq, D, device="cuda", dtype_code=BF16, stream=None):
    """Empty online-softmax state: o [B,S,Hq,D] = 0, m, l [B,Hq,S] = -inf, 0."""
    o = torch.empty((B, S, Hq, D), dtype=torch.float32, device=device)
    m = torch.empty((B, Hq, S), dtype=torch.float32, device=device)
    l = torch.empty((B, Hq, S), dtype=torch.float32, device=device)
    shp = Shape(B, S, S, Hq, Hq, D, dtype_code, 1.0)
    _check(lib().ra_state_init(shp, _ptr(o), _ptr(m), _ptr(l), _stream(stream)), "ra_state_init")
    return o, m, l


def block_attn(q, k, v, q_pos, k_pos, causal, o, m, l, scale=None, work=None, stream=None):
    """Fold the attention of q to (k, v) into the state (o, m, l) in place.
    ``work``: optional int64 CUDA tensor of 4 counters, added to."""
    _contig(q, k, v, o, m, l)
    if q_pos.dtype != torch.int32 or k_pos.dtype != torch.int32:
        raise TypeError("positions must be int32")
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    st = lib().ra_block_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(q_pos), _ptr(k_pos), int(bool(causal)),
                             _shape(q, k, scale), _ptr(o), _ptr(m), _ptr(l), _ptr(work),
                             _stream(stream))
    _check(st, "ra_block_attn")


def lse_merge(outs, ms, ls, out_dtype=torch.bfloat16, stream=None):
    """Merge partial states (lists of o [B,S,Hq,D], m, l [B,Hq,S]) into
    (out [B,S,Hq,D] in out_dtype, lse [B,Hq,S])."""
    P = len(outs)
    _contig(*outs, *ms, *ls)
    B, S, Hq, D = outs[0].shape
    out = torch.empty((B, S, Hq, D), dtype=out_dtype, device=outs[0].device)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=outs[0].device)
    arr = ctypes.c_void_p * max(P, 1)
    po = arr(*[t.data_ptr() for t in outs])
    pm = arr(*[t.data_ptr() for t in ms])
    pl = arr(*[t.data_ptr() for t in ls])
    shp = Shape(B, S, S, Hq, Hq, D, BF16 if out_dtype == torch.bfloat16 else F32, 1.0)
    st = lib().ra_lse_merge(P, ctypes.cast(po, _P), ctypes.cast(pm, _P), ctypes.cast(pl, _P), shp,
                            _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "ra_lse_merge")
    return out, lse


def schedule(c):
    t = (ctypes.c_int32 * (c * c))()
    _check(lib().ra_schedule(int(c), t), "ra_schedule")
    return [[t[s * c + i] for i in range(c)] for s in range(c)]


def shard_positions(S, c, layout):
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    t = (ctypes.c_int32 * max(S, 1))()
    _check(lib().ra_shard_positions(int(S), int(c), lay, t), "ra_shard_positions")
    return [t[i] for i in range(S)]


def work_expected(S, c, layout, causal):
    """Per (rank, step) expected work of one batch and head from the host
    scheduler: list[rank][step] = (pairs, full, partial, skipped)."""
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    w = (Work * (c * c))()
    _check(lib().ra_work_expected(int(S), int(c), lay, int(bool(causal)), w), "ra_work_expected")
    return [[(w[i * c + t].pairs, w[i * c + t].tiles_full, w[i * c + t].tiles_partial,
              w[i * c + t].tiles_skipped) for t in range(c)] for i in range(c)]


NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def ring_forward_noalloc(q, k, v, c, layout="zigzag", causal=True, mode="fused", scale=None,
                         out=None, lse=None, stream=None):
    """ring_forward through ra_ring_forward_noalloc: for callers that cannot
    allocate device memory when attention runs, the library uses its own fixed
    64 MiB scratch array instead of a workspace.  ``out`` and ``lse`` may be
    passed in (then nothing at all is allocated by this call)."""
    _contig(q, k, v)
    lay = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    md = MODES[mode] if isinstance(mode, str) else int(mode)
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=q.device)
    st = lib().ra_ring_forward_noalloc(_ptr(q), _ptr(k), _ptr(v), _shape(q, k, scale), int(c), lay,
                                       int(bool(causal)), md, _dtype_code(out), _ptr(out), _ptr(lse),
                                       _stream(stream))
    _check(st, "ra_ring_forward_noalloc")
    return out, lse


def device_error(stream=None):
    """Synchronise and read/clear the device error word; raises on a timeout."""
    _check(lib().ra_device_error(_stream(stream)), "device wait")


def selftest_wait_timeout(limit_us=20000, stream=None, leave_pending=False):
    """Run the device-timeout self-test: a bounded wait on a barrier that
    nothing arrives on.  Returns the status (TIMEOUT when the path works).
    With leave_pending the error stays set, as after a real timeout, until
    device_error() reads and clears it."""
    return int(lib().ra_selftest_wait_timeout(int(limit_us), 1 if leave_pending else 0,
                                              _stream(stream)))
