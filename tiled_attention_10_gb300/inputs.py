"""Seeded synthetic inputs for the FlashAttention forward pass.

This module holds no attention arithmetic.  It draws Q, K and V, casts them
to the storage type (round-to-nearest-even), quantises to FP8 E4M3 with a
per-tensor amax descale, and lays them out as BNSD [B, H, S, D] or
BSND [B, S, H, D].  Both the CUDA path and the float64 oracle consume exactly
the bytes produced here.

Optional NaN poisoning: the tensor is carved out of a larger buffer whose tail
(``pad_rows`` rows of the innermost [H, D] or [D] block) holds NaN bit patterns,
so any read past the last valid row would poison the result.  The Hygon
retrospective (defects 2 and 3) describes exactly this failure: garbage read
from past the tail tile turns 0 * NaN into NaN inside the accumulator.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

E4M3_MAX = 448.0

# NaN bit patterns of each storage type.
_NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "e4m3": 0x7F}
TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}
OUT_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.bfloat16}


@dataclasses.dataclass
class Workload:
    """One synthetic problem: shape, storage type, layout, mask and value recipe."""
    name: str
    B: int
    H: int
    S_q: int
    S_kv: int
    D: int
    dtype: str          # "f16" | "bf16" | "e4m3"
    layout: str         # "BNSD" | "BSND"
    causal: bool
    std: float = 1.0
    scale: Optional[float] = None   # default 1/sqrt(D)
    poison: bool = False            # NaN-poisoned memory past the valid rows
    seed: int = 0
    H_kv: Optional[int] = None      # key/value heads (grouped-query attention); default H
    split: bool = False             # run through the split-KV entry point
    bwd: bool = False               # a backward-pass workload (gradients of the forward)

    @property
    def kv_heads(self) -> int:
        return self.H if self.H_kv is None else self.H_kv

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """Nominal attention FLOPs: 4*B*H*S_q*S_kv*D, halved when causal; a
        backward pass counts 2.5 times that (five products of the forward's
        size: S recomputed, dP, dV, dK, dQ)."""
        f = 4.0 * self.B * self.H * self.S_q * self.S_kv * self.D
        f = f / 2 if self.causal else f
        return 2.5 * f if self.bwd else f

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "H_kv": self.kv_heads,
                "S_q": self.S_q,
                "S_kv": self.S_kv, "D": self.D, "dtype": self.dtype, "layout": self.layout,
                "causal": self.causal, "scale": self.softmax_scale,
                "values": f"iid N(0,{self.std}^2), seed {self.seed}"
                          + (", per-tensor amax e4m3" if self.dtype == "e4m3" else "")
                          + (", NaN-poisoned tail" if self.poison else ""),
                **({"pass": "backward (dQ, dK, dV from O, dO, lse)"} if self.bwd else {})}


# The five workloads the method is measured and checked on.
WORKLOADS = {
    "fp16_1x8x512x64": Workload("fp16_1x8x512x64", 1, 8, 512, 512, 64, "f16", "BNSD", False,
                                scale=1.0 / 8.0),
    "bf16_bsnd_causal_2x16x4097x64": Workload("bf16_bsnd_causal_2x16x4097x64", 2, 16, 4097,
                                              4097, 64, "bf16", "BSND", True, scale=1.0 / 8.0,
                                              poison=True),
    "bf16_4x32x4096x128": Workload("bf16_4x32x4096x128", 4, 32, 4096, 4096, 128, "bf16",
                                   "BNSD", False),
    "fp8_causal_1x32x8192x128": Workload("fp8_causal_1x32x8192x128", 1, 32, 8192, 8192, 128,
                                         "e4m3", "BNSD", True),
    "bf16_causal_16x64x16384x128": Workload("bf16_causal_16x64x16384x128", 16, 64, 16384,
                                            16384, 128, "bf16", "BNSD", True, std=0.5),
}
HEADLINE = "bf16_4x32x4096x128"

# Further workloads for the steps beyond the measured five (same recipe).
EXTRA_WORKLOADS = {
    # grouped-query attention: 32 query heads on 8 key/value heads
    "bf16_gqa_4x32kv8x4096x128": Workload("bf16_gqa_4x32kv8x4096x128", 4, 32, 4096, 4096, 128,
                                          "bf16", "BNSD", False, H_kv=8),
    "bf16_gqa_causal_1x64kv8x8192x128": Workload("bf16_gqa_causal_1x64kv8x8192x128", 1, 64, 8192,
                                                 8192, 128, "bf16", "BSND", True, H_kv=8),
    # few heads, short queries, long keys: split-KV fills the GPU
    "bf16_splitkv_1x8x512x16384x128": Workload("bf16_splitkv_1x8x512x16384x128", 1, 8, 512, 16384,
                                               128, "bf16", "BNSD", False, split=True),
}
# Backward pass: the training configuration of the Ascend page (32 heads,
# head dim 128, causal, bf16) at the forward's 4 x 4096 tokens, and the
# forward's non-causal shape.
BWD_WORKLOADS = {
    "bf16_bwd_causal_4x32x4096x128": Workload("bf16_bwd_causal_4x32x4096x128", 4, 32, 4096, 4096,
                                              128, "bf16", "BNSD", True, bwd=True),
    "bf16_bwd_4x32x4096x128": Workload("bf16_bwd_4x32x4096x128", 4, 32, 4096, 4096, 128, "bf16",
                                       "BNSD", False, bwd=True),
}
EXTRA_WORKLOADS.update(BWD_WORKLOADS)
ALL_WORKLOADS = {**WORKLOADS, **EXTRA_WORKLOADS}


def shape_of(layout: str, B: int, H: int, S: int, D: int):
    return (B, H, S, D) if layout == "BNSD" else (B, S, H, D)


def _draw(shape, std, seed, device, chunk=1 << 28):
    """float32 N(0, std^2) samples from a generator seeded with `seed`."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty(shape, dtype=torch.float32, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk):       # bounded temporaries on big tensors
        e = min(flat.numel(), s + chunk)
        flat[s:e].normal_(0.0, std, generator=g)
    return out


def _cast(x32: torch.Tensor, dtype: str):
    """Storage cast; for e4m3 also the per-tensor descale (amax / 448)."""
    if dtype != "e4m3":
        return x32.to(TORCH_DTYPE[dtype]), 1.0
    amax = float(x32.abs().max())
    descale = amax / E4M3_MAX if amax > 0 else 1.0
    # torch's float8 cast does not saturate: clamp first so nothing becomes NaN.
    q = (x32 / descale).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q, descale


def poisoned_like(shape, dtype: str, device, pad_elems: int):
    """A flat buffer of numel(shape) + pad_elems elements filled with NaN bits,
    and a contiguous view of its first numel(shape) elements."""
    n = math.prod(shape)
    if dtype == "e4m3":
        buf = torch.full((n + pad_elems,), _NAN_BITS[dtype], dtype=torch.uint8, device=device)
    else:
        buf = torch.full((n + pad_elems,), _NAN_BITS[dtype], dtype=torch.int16, device=device)
    buf = buf.view(TORCH_DTYPE[dtype])
    return buf, buf[:n].view(shape)


@dataclasses.dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    descale: tuple          # (dq, dk, dv); (1, 1, 1) unless e4m3
    buffers: tuple          # the backing buffers (padded when poisoned)


def make_inputs(w: Workload, device="cpu", pad_rows: int = 128) -> Inputs:
    """Draw Q, K, V for workload `w` (seeds 3*seed + 0/1/2) on `device`."""
    qs = shape_of(w.layout, w.B, w.H, w.S_q, w.D)
    ks = shape_of(w.layout, w.B, w.kv_heads, w.S_kv, w.D)
    tensors, descales, bufs = [], [], []
    for i, shp in enumerate((qs, ks, ks)):
        x32 = _draw(shp, w.std, 3 * w.seed + i, device)
        x, ds = _cast(x32, w.dtype)
        del x32
        if w.poison:
            pad = pad_rows * (w.H if i == 0 else w.kv_heads) * w.D
            buf, view = poisoned_like(shp, w.dtype, device, pad)
            view.copy_(x)
            x = view
        else:
            buf = x
        tensors.append(x)
        descales.append(ds)
        bufs.append(buf)
    return Inputs(tensors[0], tensors[1], tensors[2], tuple(descales), tuple(bufs))


def sample_rows(w: Workload, n: int, seed: int = 0):
    """n (b, h, i) triples: the two corners plus n-2 uniform draws."""
    import numpy as np
    rng = np.random.default_rng(seed)
    rows = [(0, 0, 0), (w.B - 1, w.H - 1, w.S_q - 1)]
    for _ in range(max(0, n - 2)):
        rows.append((int(rng.integers(w.B)), int(rng.integers(w.H)), int(rng.integers(w.S_q))))
    return np.asarray(rows[:n], dtype=np.int64)


def make_dout(w: Workload, device="cpu") -> torch.Tensor:
    """Upstream gradient dO for a backward workload: iid N(0, 1) in Q's shape,
    layout and storage type, from its own seed (1000 + the workload's)."""
    wd = dataclasses.replace(w, name=w.name + "/dO", S_kv=w.S_q, H_kv=None, seed=1000 + w.seed,
                             std=1.0, split=False, bwd=False)
    return make_inputs(wd, device=device).q
