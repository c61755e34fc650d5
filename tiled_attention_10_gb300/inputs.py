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
import itertools
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
    # the forward of the training configuration (32 heads, head dim 128,
    # causal, bf16) at 4 x 4096 tokens: the pass the backward workload follows
    "bf16_causal_4x32x4096x128": Workload("bf16_causal_4x32x4096x128", 4, 32, 4096, 4096, 128,
                                          "bf16", "BNSD", True),
    # one batch of the 16 x 64 x 16384 causal workload (same shape per head,
    # values N(0, 0.5^2)): small enough for a profiler capture of one launch
    "bf16_causal_1x64x16384x128": Workload("bf16_causal_1x64x16384x128", 1, 64, 16384, 16384,
                                           128, "bf16", "BNSD", True, std=0.5),
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


# ---------------------------------------------------------------------------
# Packed variable-length batches (varlen / paged K/V).
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class PackedWorkload:
    """A batch of sequences packed row after row: queries [total_q, H, D];
    keys and values packed the same way (page_size 0) or in a paged cache
    [num_pages, page_size, H_kv, D] whose pages are shuffled (seeded)."""
    name: str
    seq_q: tuple
    seq_k: tuple
    H: int
    H_kv: int
    D: int
    dtype: str
    causal: int             # 0 none, 1 top-left, 2 bottom-right
    page_size: int = 0      # 0: contiguous packed K/V
    seed: int = 0
    std: float = 1.0
    n_splits: int = 1       # paged: keys of each unit split this many ways, then merged;
                            # 0: as many as fa_fwd_paged_split_plan picks

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def decode(self) -> bool:
        return all(n == 1 for n in self.seq_q)

    def visible_pairs(self) -> int:
        """(query, key) pairs the masks leave, summed over sequences."""
        tot = 0
        for sq, sk in zip(self.seq_q, self.seq_k):
            if self.causal == 0:
                tot += sq * sk
                continue
            off = 0 if self.causal == 1 else sk - sq
            for i in range(sq):
                tot += max(0, min(sk, i + off + 1))
        return tot

    @property
    def flops(self) -> float:
        """4 * D * H FLOPs per visible (query, key) pair."""
        return 4.0 * self.D * self.H * self.visible_pairs()

    @property
    def kv_bytes(self) -> int:
        eb = 1 if self.dtype == "e4m3" else 2
        return 2 * sum(self.seq_k) * self.H_kv * self.D * eb

    def describe(self) -> dict:
        return {"workload": self.name, "n_seqs": len(self.seq_q), "total_q": sum(self.seq_q),
                "total_k": sum(self.seq_k), "seq_q": f"{min(self.seq_q)}..{max(self.seq_q)}",
                "seq_k": f"{min(self.seq_k)}..{max(self.seq_k)}", "H": self.H,
                "H_kv": self.H_kv, "D": self.D, "dtype": self.dtype,
                "causal": ["none", "top-left", "bottom-right"][self.causal],
                "page_size": self.page_size or "contiguous",
                **({"n_splits": self.n_splits or "planned"} if self.n_splits != 1 else {}),
                "values": f"iid N(0,{self.std}^2), seed {self.seed}"}


def _log_uniform_lengths(n, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    u = torch.rand(n, generator=g, dtype=torch.float64)
    return tuple(int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo)))))
                 for x in u)


PACKED_WORKLOADS = {
    # training-style packed batch: 32 sequences, lengths log-uniform in [512, 8192]
    "bf16_varlen_causal_32seq_512-8192_h32x128": PackedWorkload(
        "bf16_varlen_causal_32seq_512-8192_h32x128", _log_uniform_lengths(32, 512, 8192, 11),
        _log_uniform_lengths(32, 512, 8192, 11), 32, 32, 128, "bf16", 1),
    # prefix prefill against a paged cache of 64-token pages (the page size of
    # the Hygon retrospective's defect 11): 1024 new tokens after 7168 cached
    "bf16_paged_prefill_8x1024of8192_p64_h32kv8": PackedWorkload(
        "bf16_paged_prefill_8x1024of8192_p64_h32kv8", (1024,) * 8, (8192,) * 8, 32, 8, 128,
        "bf16", 2, page_size=64),
    # decode: one new token per sequence, cached lengths log-uniform in [1K, 32K];
    # keys split per sequence and merged (fa_fwd_paged_split), as many ways as
    # fa_fwd_paged_split_plan picks (2 here)
    "bf16_paged_decode_128seq_1k-32k_p64_h32kv8": PackedWorkload(
        "bf16_paged_decode_128seq_1k-32k_p64_h32kv8", (1,) * 128,
        _log_uniform_lengths(128, 1024, 32768, 12), 32, 8, 128, "bf16", 2, page_size=64,
        n_splits=0),
    # the same decode at a quarter of the cache (about 1 GB of K/V): the size
    # the detailed profiler captures are taken on (5 splits planned)
    "bf16_paged_decode_32seq_1k-32k_p64_h32kv8": PackedWorkload(
        "bf16_paged_decode_32seq_1k-32k_p64_h32kv8", (1,) * 32,
        _log_uniform_lengths(32, 1024, 32768, 12), 32, 8, 128, "bf16", 2, page_size=64,
        n_splits=0),
}


@dataclasses.dataclass
class PackedInputs:
    q: torch.Tensor
    k: torch.Tensor           # packed [total_k, H_kv, D] or cache [pages, page_size, H_kv, D]
    v: torch.Tensor
    cu_q: torch.Tensor        # int32 [n_seqs + 1]
    cu_k: Optional[torch.Tensor]
    seqused_k: Optional[torch.Tensor]
    block_table: Optional[torch.Tensor]
    descale: tuple


def make_packed_inputs(w: PackedWorkload, device="cpu") -> PackedInputs:
    """Seeded inputs of a packed workload (no attention arithmetic here)."""
    tq, tk = sum(w.seq_q), sum(w.seq_k)
    cu_q = torch.tensor([0] + list(itertools.accumulate(w.seq_q)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(itertools.accumulate(w.seq_k)), dtype=torch.int32)
    q, dq = _cast(_draw((tq, w.H, w.D), w.std, 3 * w.seed, device), w.dtype)
    k, dk = _cast(_draw((tk, w.H_kv, w.D), w.std, 3 * w.seed + 1, device), w.dtype)
    v, dv = _cast(_draw((tk, w.H_kv, w.D), w.std, 3 * w.seed + 2, device), w.dtype)
    if not w.page_size:
        return PackedInputs(q, k, v, cu_q.to(device), cu_k.to(device), None, None, (dq, dk, dv))
    ps = w.page_size
    n_pages = [max(1, -(-n // ps)) for n in w.seq_k]
    total_pages = sum(n_pages)
    g = torch.Generator().manual_seed(1000 + w.seed)
    phys = torch.randperm(total_pages, generator=g).tolist()
    table = torch.zeros(len(w.seq_k), max(n_pages), dtype=torch.int32)
    caches = []
    for src in (k, v):
        cache = torch.zeros((total_pages, ps, w.H_kv, w.D), dtype=src.dtype, device=device)
        nxt = 0
        for s, n in enumerate(w.seq_k):
            base = int(cu_k[s])
            for pg in range(n_pages[s]):
                pid = phys[nxt]
                nxt += 1
                table[s, pg] = pid
                lo, hi = base + pg * ps, base + min(n, (pg + 1) * ps)
                if hi > lo:
                    cache[pid, : hi - lo] = src[lo:hi]
        caches.append(cache)
    seqused = torch.tensor(w.seq_k, dtype=torch.int32)
    return PackedInputs(q, caches[0], caches[1], cu_q.to(device), None, seqused.to(device),
                        table.to(device), (dq, dk, dv))
