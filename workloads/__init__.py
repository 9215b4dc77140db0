"""Seeded synthetic workloads shared by the tests, the smoke check and the bench.

This module only draws random inputs and names the five workload shapes; it
holds none of the attention arithmetic, so both the CPU oracle and the CUDA
path can be fed from it without sharing any of the method's code.

Generator (the pages fix none): ``torch.Generator('cpu').manual_seed(seed)``
draws Q, K, V in that order as float32 N(0, 1) of shape [B, S, H, D]; the
workload's scaling is applied in float32; the tensors are then rounded to the
workload's dtype.  Oracle and GPU read the same rounded tensors.

Workloads (from the description of the five test configurations):
  tiny     S=256,   c=4,  contiguous, non-causal, B=1, Hq=2,  Hkv=1, D=64,  fp32
  gqa4k    S=4096,  c=4,  zig-zag,    causal,     B=1, Hq=8,  Hkv=2, D=128, bf16, x 1/sqrt(128)
  s32k     S=32768, c=8,  contiguous and zig-zag, causal, B=1, Hq=32, Hkv=8, D=128, bf16
  s128k    S=131072,c=16, zig-zag,    causal,     B=1, Hq=16, Hkv=1, D=128, bf16
  stress   S=65536, c=8,  zig-zag,    causal,     B=2, Hq=16, Hkv=2, D=128, bf16,
           Q and K x sqrt(30) (logits ~ N(0, 30^2) after the 1/sqrt(D) scale),
           1% of key rows (per batch and KV head, drawn without replacement
           from the second half of the sequence) get +50 added to every
           element.
"""

from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    S: int
    c: int
    layouts: tuple
    causal: bool
    B: int
    Hq: int
    Hkv: int
    D: int
    dtype: str          # "bf16" or "f32"
    seed: int
    qkv_scale: float = 1.0
    qk_scale: float = 1.0
    offset_frac: float = 0.0
    offset_value: float = 0.0

    @property
    def scale(self) -> float:
        """Softmax scale passed to the kernels and the oracle: 1/sqrt(D)."""
        return 1.0 / math.sqrt(self.D)

    def flops(self) -> int:
        """Algorithmic FLOP of one full attention: 4*B*Hq*D per visible pair."""
        pairs = self.S * (self.S + 1) // 2 if self.causal else self.S * self.S
        return 4 * self.B * self.Hq * self.D * pairs

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 256, 4, ("contiguous",), False, 1, 2, 1, 64, "f32", 0),
    "gqa4k": Workload("gqa4k", 4096, 4, ("zigzag",), True, 1, 8, 2, 128, "bf16", 1,
                      qkv_scale=1.0 / math.sqrt(128.0)),
    "s32k": Workload("s32k", 32768, 8, ("contiguous", "zigzag"), True, 1, 32, 8, 128, "bf16", 2),
    "s128k": Workload("s128k", 131072, 16, ("zigzag",), True, 1, 16, 1, 128, "bf16", 3),
    "stress": Workload("stress", 65536, 8, ("zigzag",), True, 2, 16, 2, 128, "bf16", 4,
                       qk_scale=math.sqrt(30.0), offset_frac=0.01, offset_value=50.0),
}


def torch_dtype(name: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def make_inputs(w: Workload):
    """Return (q, k, v) CPU tensors in the workload dtype, layout [B, S, H, D],
    plus the sorted offset key rows per (batch, kv head) (empty if none)."""
    g = torch.Generator(device="cpu").manual_seed(w.seed)
    q = torch.randn((w.B, w.S, w.Hq, w.D), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.S, w.Hkv, w.D), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.S, w.Hkv, w.D), generator=g, dtype=torch.float32)
    if w.qkv_scale != 1.0:
        q.mul_(w.qkv_scale)
        k.mul_(w.qkv_scale)
        v.mul_(w.qkv_scale)
    if w.qk_scale != 1.0:
        q.mul_(w.qk_scale)
        k.mul_(w.qk_scale)
    offsets = {}
    if w.offset_frac > 0:
        n_off = math.ceil(w.offset_frac * w.S)
        half = w.S // 2
        for b in range(w.B):
            for h in range(w.Hkv):
                rows = torch.randperm(w.S - half, generator=g)[:n_off] + half
                rows, _ = torch.sort(rows)
                k[b, rows, h, :] += w.offset_value
                offsets[(b, h)] = rows
    dt = torch_dtype(w.dtype)
    return q.to(dt), k.to(dt), v.to(dt), offsets


def small_case(S, c, layout, causal, B=1, Hq=4, Hkv=2, D=128, dtype="bf16", seed=11):
    """An ad-hoc workload for parity tests (ragged, odd head counts, ...)."""
    return Workload(f"case_S{S}_c{c}_{layout}", S, c, (layout,), causal, B, Hq, Hkv, D, dtype, seed)
