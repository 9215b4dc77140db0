#!/usr/bin/env python3
"""Causal ring-attention throughput on GB300.

One step = one full ring attention (ra_ring_prepare + ra_ring_attend: shard
pack, heavy-first block order, all c ring steps and the normalisation) over
the s128k workload: S = 131072 tokens, c = 16 virtual ranks, zig-zag split,
causal, batch 1, 16 query heads / 1 KV head, head dim 128, bf16.  The metric
is algorithmic causal TFLOP/s: 4 * B * Hq * D * S(S+1)/2 FLOP per step over
the device time of the step.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own independent ring (weak scaling).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal ring-attention TFLOP/s on 1 GB300; % of dense BF16 tensor peak"
NOMINAL_BF16_DENSE_TFLOPS = 2250.0   # GB300 nominal dense bf16 (no sparsity)
L2_FLUSH_BYTES = 512 * 1024 * 1024   # > 129 MB L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="s128k")
    ap.add_argument("--layout", default=None)
    ap.add_argument("--mode", default="fused", choices=["fused", "per_step", "allgather"],
                    help="fused ring (one launch), one launch per ring step, or one step over all-gathered keys")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--overlap-study", action="store_true",
                    help="time the ring with real K/V rotation, overlapped and not")
    ap.add_argument("--lse-merge", type=int, default=0, metavar="P",
                    help="time ra_lse_merge of P partial states of the workload's shape instead")
    ap.add_argument("--decode", action="store_true",
                    help="time decode over the sharded keys (one new token per step) instead")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, world, device=None):
    """The largest of every rank's value (the job waits for the slowest rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(flop_per_rank_step, world, ms_per_step):
    """Aggregate TFLOP/s of `world` ranks that each did one step of
    `flop_per_rank_step` FLOP in `ms_per_step` (the max over ranks)."""
    return world * flop_per_rank_step / (ms_per_step * 1e-3) / 1e12


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_traffic(kernel_src):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "attn_fwd_pair_s128k_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        src = open(os.path.join(ROOT, "context_exact_attention_ra_gb300", "csrc", kernel_src), "rb").read()
        if d.get("kernel_sha256") == hashlib.sha256(src).hexdigest():
            return int(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, enabled=True):
        self.index = index
        self.proc = None
        self.path = None
        if not enabled:
            return
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def cpu_baseline(w, layout, seconds, q, k, v):
    """The float64 oracle on this host's cores over a bounded sample of query
    rows of the same workload; throughput in algorithmic TFLOP/s."""
    import numpy as np
    import oracle

    import torch

    rng = np.random.default_rng(w.seed)
    pos = np.arange(w.S)
    h, g = 0, 0                      # query head 0 reads key/value head 0
    kk = k[:, :, g:g + 1].to(torch.float64).numpy()
    vv = v[:, :, g:g + 1].to(torch.float64).numpy()
    done_flop = 0.0
    rows_done = 0
    t0 = time.perf_counter()
    batch = 32
    while time.perf_counter() - t0 < seconds:
        rows = np.sort(rng.integers(0, w.S, size=batch))
        qq = q[:, torch.as_tensor(rows), h:h + 1].to(torch.float64).numpy()
        oracle.attention_reference(qq, kk, vv, pos[rows], pos, w.causal, w.scale)
        vis = (rows + 1) if w.causal else np.full(rows.size, w.S)
        done_flop += 4.0 * w.D * float(vis.sum()) * w.B
        rows_done += rows.size * w.B
    el = time.perf_counter() - t0
    cores = os.cpu_count()
    return {"value": done_flop / el / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows_done} random query rows (1 head, float64 full-row masked softmax) of the "
                      f"{w.name} workload in {el:.1f} s; BLAS threads default to all {cores} cores",
            "elapsed_s": el, "rows": rows_done}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, on host cores."""
    import torch
    from workloads import WORKLOADS, make_inputs

    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    layout = args.layout or w.layouts[0]
    q, k, v, _ = make_inputs(w)
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(w, layout, min(per_step, 2.0), q, k, v)
    vals = [cpu_baseline(w, layout, per_step, q, k, v) for _ in range(args.steps)]
    val = statistics.median(x["value"] for x in vals)
    flop = w.flops()
    # A step is one bounded sample of the workload (random query rows for a
    # fixed CPU time): its measured wall time is the step time.  The time the
    # whole workload would take at the same rate is an extrapolation, reported
    # under its own key.
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.median(x["elapsed_s"] for x in vals) * 1e3,
        "ms_per_step_extrapolated": flop / (val * 1e12) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{w.name}: S={w.S} c={w.c} {layout} causal B={w.B} "
                                                    f"Hq={w.Hq} Hkv={w.Hkv} D={w.D} {w.dtype}",
                                        "sample": f"each step: random query rows of the workload for "
                                                  f"{per_step:.1f} s of CPU time "
                                                  f"(median {statistics.median(x['rows'] for x in vals)} rows); "
                                                  f"ms_per_step_extrapolated = the whole workload at that "
                                                  f"rate (extrapolated, not measured)"},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": vals[0]["cores"], "kind": "oracle",
                         "sample": vals[0]["sample"] + "; full-workload time extrapolated"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist

    import context_exact_attention_ra_gb300 as ra
    from workloads import WORKLOADS, make_inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    w = WORKLOADS[args.workload]
    layout = args.layout or w.layouts[0]
    q, k, v, _ = make_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    shp = ra.Shape(w.B, w.S, w.S, w.Hq, w.Hkv, w.D, ra.BF16 if w.dtype == "bf16" else ra.F32, w.scale)
    lay = ra.LAYOUTS[layout]
    md = ra.MODES[args.mode]
    ws = torch.empty(ra.ring_workspace_size(shp, w.c, lay, md), dtype=torch.uint8, device=dev)
    out = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        ra.ring_prepare(qd, kd, vd, w.c, lay, ws, scale=w.scale)
        ra.ring_attend(shp, w.c, lay, w.causal, md, out, lse, ws)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    ra.device_error()
    # ra_ring_prepare: pack, tile ranges, heavy-first block order (every
    # workload here has more than one query block); ra_ring_attend: one
    # launch, or one launch per ring step in per-step mode
    prep_launches = 3
    launches_per_step = prep_launches + (w.c if md == ra.MODE_PER_STEP else 1)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()   # L2 flush between timed steps (outside the events)
        e0, e1, e2 = ev[i]
        e0.record(stream)
        ra.ring_prepare(qd, kd, vd, w.c, lay, ws, scale=w.scale)
        e1.record(stream)
        ra.ring_attend(shp, w.c, lay, w.causal, md, out, lse, ws)
        e2.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ra.device_error()
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    attend_ms = [b.elapsed_time(c) for _, b, c in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    flop = w.flops()
    value = whole_job_throughput(flop, world, ms_per_step)

    peaks, peak_kind = load_peaks()
    attn_ms = statistics.mean(attend_ms)
    achieved = flop / (attn_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": kernel_traffic("attn_pair_sm103.cu") if md == ra.MODE_FUSED else None,
            "kernel": {ra.MODE_FUSED: "attn_fwd_pair_kernel (CTA pairs, D = 128)",
                       ra.MODE_ALLGATHER: "attn_fwd_pair_kernel (one step over the gathered keys)"}.get(
                           md, "attn_fwd_pair_kernel (one launch per ring step)"),
            "peak_source": f"{peak_kind} bf16_tflops (burst)",
            "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained", peak)),
            "frac_of_nominal_dense": achieved / NOMINAL_BF16_DENSE_TFLOPS}

    # The work the ring did, counted on the GPU by one more call outside the
    # timed region: the tiles executed (diagonal tiles computed whole) next to
    # the algorithmic FLOP, the load imbalance over the ranks, and the K/V bytes
    # a ring over real devices would pass (derived, not timed).
    _, _, info = ra.ring_forward(qd, kd, vd, w.c, layout, w.causal, args.mode, scale=w.scale, report=True)
    ra.device_error()
    tiles = sum(x["full"] + x["partial"] for row in info["per_rank_step"] for x in row)
    work = {"algorithmic_flop": int(info["algorithmic_flop"]),
            "executed_tiles": int(tiles), "tile": "128 query rows x 128 keys of one (batch, head)",
            "executed_tile_flop": int(4 * w.D * 128 * 128 * tiles),
            "imbalance_pairs": info["imbalance_pairs"], "imbalance_tiles": info["imbalance_tiles"],
            "ring_kv_bytes": int(info["ring_kv_bytes"]), "ring_kv_bytes_sent": int(info["ring_kv_bytes_sent"])}

    # end to end through the C ABI with host buffers (copies inside the call)
    e2e = None
    if args.e2e_steps > 0:
        qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
        oh = torch.empty_like(qh).pin_memory()
        lh = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32).pin_memory()
        need = ra.hostio_workspace_size(shp, w.c, lay, md)
        del ws
        wsh = torch.empty(need, dtype=torch.uint8, device=dev)
        ra.ring_forward_hostio(qh, kh, vh, w.c, layout, w.causal, args.mode, w.scale, oh, lh, wsh)
        times = []
        for _ in range(args.e2e_steps):
            flush.zero_()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ra.ring_forward_hostio(qh, kh, vh, w.c, layout, w.causal, args.mode, w.scale, oh, lh, wsh)
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        e2e_ms = max_over_ranks(statistics.mean(times), world, dev)
        bi = (q.numel() + k.numel() + v.numel()) * q.element_size()
        bo = oh.numel() * oh.element_size() + lh.numel() * 4
        e2e = {"value": whole_job_throughput(flop, world, e2e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, layout, args.cpu_seconds, q, k, v)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic",
            "config": {"workload": f"{w.name}: S={w.S} c={w.c} {layout} causal={w.causal} B={w.B} "
                                   f"Hq={w.Hq} Hkv={w.Hkv} D={w.D} {w.dtype}",
                       "mode": args.mode, "l2": "flushed (512 MiB write) before every timed step",
                       "flop_per_step": flop, "parallelism": f"{w.c} virtual ranks per GPU"},
            "pct_dense_bf16_peak": {"of_measured": value / world / peak * 100,
                                    "of_nominal_2250": value / world / NOMINAL_BF16_DENSE_TFLOPS * 100},
            "roofline": roof,
            "work": work,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "attend_ms": attn_ms,
            "prepare_ms": statistics.mean(a.elapsed_time(b) for a, b, _ in ev),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_decode(args, rank, world, local):
    """Decode over distributed keys and values: one new token's 16 query heads
    against the s128k keys and values held in 16 zig-zag shards (split-K
    partials per shard piece + merge).  HBM-bound: the algorithmic bytes of a
    step are one read of K and V plus q, out and lse."""
    import torch

    import context_exact_attention_ra_gb300 as ra
    from workloads import WORKLOADS

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    layout = args.layout or w.layouts[0]
    g = torch.Generator().manual_seed(w.seed)
    k = torch.randn((w.B, w.S, w.Hkv, w.D), generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn((w.B, w.S, w.Hkv, w.D), generator=g).to(torch.bfloat16).to(dev)
    q = torch.randn((w.B, 1, w.Hq, w.D), generator=g).to(torch.bfloat16).to(dev)
    q_pos = torch.tensor([w.S - 1], dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = torch.empty((w.B, 1, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device=dev)
    shp = ra.Shape(w.B, 1, w.S, w.Hq, w.Hkv, w.D, ra.BF16, w.D ** -0.5)
    ws = torch.empty(max(int(ra.lib().ra_decode_workspace_size(shp, w.c, ra.LAYOUTS[layout])), 256),
                     dtype=torch.uint8, device=dev)

    def call(stream=None):
        ra.decode_forward(q, q_pos, k, v, w.c, layout, True, out=out, lse=lse, workspace=ws, stream=stream)

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        call()
    ra.device_error()

    def timed(fn, clean=True):
        """Median step time.  Before every step (outside the events) L2 is
        flushed by writing a 512 MiB buffer; with `clean` the buffer is then
        also read, so that L2 holds clean lines and the step's reads do not
        first write back the flush's dirty lines (which would double the DRAM
        traffic of an HBM-bound step)."""
        times = []
        for _ in range(args.steps):
            flush.zero_()
            if clean:
                flush.sum()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        return statistics.median(times)

    # The call is issued from the host while the L2 flush still runs on the
    # device (about 0.15 ms of work), so its two launches sit in the queue
    # when the events around them are reached: the events time the device's
    # work for one call, the launch gap between the two kernels included.
    ms = timed(call)
    ms_dirty = timed(call, clean=False)
    ra.device_error()
    # The same call captured once in a CUDA graph and replayed between the
    # events; and a graph holding one trivial kernel, timed the same way: the
    # device-side latency of a graph launch, paid by any graph however small.
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            call(side)
    stream.wait_stream(side)
    tiny = torch.zeros(1, device=dev)
    tiny_graph = torch.cuda.CUDAGraph()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(tiny_graph, stream=side):
            tiny.add_(1.0)
    stream.wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    ra.device_error()
    graph_ms = timed(graph.replay)
    tiny_graph_ms = timed(tiny_graph.replay)
    ra.device_error()
    # For scale: the device reading the same K and V bytes with two library
    # reductions (torch.sum over K, then over V), timed the same way.
    read_ms = timed(lambda: (k.sum(), v.sum()))
    nbytes = 2 * k.numel() * k.element_size() + 2 * q.numel() * q.element_size() + w.B * w.Hq * 4
    peaks, kind = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "decode over distributed KV: achieved GB/s (one token, K/V read once)",
        "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"decode: 1 token, {w.name} keys S={w.S} c={w.c} {layout} Hq={w.Hq} "
                               f"Hkv={w.Hkv} D={w.D}",
                   "l2": "flushed before every step: 512 MiB written, then read (L2 left holding clean lines)",
                   "timing": "one decode call (two kernel launches) issued while the L2 flush still runs, "
                             "so that its launches are queued; CUDA events around it on the launching stream",
                   "graph_ms_per_step": graph_ms,
                   "gbs_graph": nbytes / (graph_ms * 1e-3) / 1e9,
                   "one_kernel_graph_ms": tiny_graph_ms,
                   "torch_sum_k_then_v_ms": read_ms,
                   "gbs_torch_sum_k_then_v": nbytes / (read_ms * 1e-3) / 1e9,
                   "ms_per_step_write_only_flush": ms_dirty,
                   "gbs_write_only_flush": nbytes / (ms_dirty * 1e-3) / 1e9},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]),
                     "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]), "traffic": None,
                     "kernel": "decode_tc_kernel + decode_merge_kernel"},
        "gpu_launches": 2 * args.steps}), flush=True)


def run_overlap_study(args, rank, world, local):
    """The tutorial's exercise C on one GPU: the ring with its K/V pass made
    real (device-to-device rotation between steps), with the copies on a
    second stream overlapped with the attention, and serialised."""
    import torch

    import context_exact_attention_ra_gb300 as ra
    from workloads import WORKLOADS, make_inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    layout = args.layout or w.layouts[0]
    q, k, v, _ = make_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    shp = ra.Shape(w.B, w.S, w.S, w.Hq, w.Hkv, w.D, ra.BF16 if w.dtype == "bf16" else ra.F32, w.scale)
    ws = torch.empty(int(ra.lib().ra_ring_rotate_workspace_size(shp, w.c, ra.LAYOUTS[layout])),
                     dtype=torch.uint8, device=dev)
    copy_stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    res = {}
    for name, fn in (("per_step", lambda: ra.ring_forward(qd, kd, vd, w.c, layout, w.causal, "per_step", scale=w.scale)),
                     ("rotate_serial", lambda: ra.ring_forward_rotate(qd, kd, vd, w.c, layout, w.causal, False,
                                                                      scale=w.scale, workspace=ws)),
                     ("rotate_overlap", lambda: ra.ring_forward_rotate(qd, kd, vd, w.c, layout, w.causal, True,
                                                                       scale=w.scale, workspace=ws,
                                                                       copy_stream=copy_stream))):
        for _ in range(args.warmup):
            fn()
        times = []
        for _ in range(args.steps):
            flush.zero_()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        res[name] = statistics.median(times)
    ra.device_error()
    kv_bytes_per_step = 2 * k.numel() * k.element_size()
    print(json.dumps({
        "metric": "ring step time with the K/V rotation overlapped vs serialised (ms per ring)",
        "unit": "ms", "steps": args.steps, "warmup": args.warmup,
        "config": {"workload": f"{w.name}: S={w.S} c={w.c} {layout} Hq={w.Hq} Hkv={w.Hkv} D={w.D}"},
        "ms": res, "overlap_saving_ms": res["rotate_serial"] - res["rotate_overlap"],
        "rotation_bytes_per_step": kv_bytes_per_step, "ring_steps": w.c,
        "flop": w.flops()}), flush=True)


def run_lse_merge(args, rank, world, local):
    """ra_lse_merge of P partial states (o fp32 [B,S,Hq,D], m, l [B,Hq,S]) of
    the workload's shape into bf16 out + lse.  HBM-bound: the algorithmic bytes
    are P*(4D + 8) per row read and 2D + 4 per row written."""
    import torch

    import context_exact_attention_ra_gb300 as ra
    from workloads import WORKLOADS

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    P = args.lse_merge
    g = torch.Generator(device=dev).manual_seed(w.seed)
    outs = [torch.randn((w.B, w.S, w.Hq, w.D), generator=g, device=dev) for _ in range(P)]
    ms = [torch.randn((w.B, w.Hq, w.S), generator=g, device=dev) * 4 for _ in range(P)]
    ls = [torch.rand((w.B, w.Hq, w.S), generator=g, device=dev) * 100 + 1 for _ in range(P)]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        ra.lse_merge(outs, ms, ls, torch.bfloat16)
    ra.device_error()
    times = []
    for _ in range(args.steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ra.lse_merge(outs, ms, ls, torch.bfloat16)
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ra.device_error()
    ms_step = statistics.median(times)
    rows = w.B * w.Hq * w.S
    nbytes = rows * (P * (4 * w.D + 8) + 2 * w.D + 4)
    peaks, kind = load_peaks()
    gbs = nbytes / (ms_step * 1e-3) / 1e9
    print(json.dumps({
        "metric": "ra_lse_merge of P partial states: achieved GB/s", "value": gbs, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "dtype": "f32 in, bf16 out", "data": "synthetic",
        "config": {"workload": f"{w.name} shape B={w.B} S={w.S} Hq={w.Hq} D={w.D}, P={P} partials",
                   "l2": "flushed before every step"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                     "frac": gbs / float(peaks["hbm_gbs"]), "traffic": None,
                     "kernel": "merge_kernel" if P > 1 else "finalize_kernel"},
        "gpu_launches": args.steps}), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.lse_merge > 0:
        run_lse_merge(args, rank, world, local)
        return
    if args.overlap_study:
        run_overlap_study(args, rank, world, local)
        return
    if args.decode:
        run_decode(args, rank, world, local)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
