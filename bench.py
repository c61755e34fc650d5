#!/usr/bin/env python
"""Benchmark of the FlashAttention forward pass (libfa_b200) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline] [--oracle-full]

One step = one fa_fwd call over the whole workload (default: bf16
B=4, H=32, S_q=S_kv=4096, D=128, BNSD, non-causal), inputs resident in HBM.
Prints one JSON line: attention TFLOP/s (4*B*H*S_q*S_kv*D FLOPs, halved when
causal) over all ranks, plus roofline, e2e (host buffers), clocks and the
float64 oracle timed on the host cores as a CPU baseline.

--impl reference times that oracle (the reference arm: a deliberately slow
CPU program) on a bounded sample of the same workload per step.
Under torchrun each rank runs its own independent shard of (batch, head)
units (weak scaling; no collective on the data path).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


FWD_SOURCES = ("fa_api.cu", "fa_kernel.cuh", "fa_ptx.cuh", "fa_tmem_io.cuh", "fa_inst_*.cu")
BWD_SOURCES = ("fa_api.cu", "fa_bwd.cuh", "fa_ptx.cuh", "fa_tmem_io.cuh", "fa_bwd_inst_*.cu")


def _code_only(text: str) -> str:
    """C++ source without its comments and with runs of white space collapsed (the kernel
    sources hold no string literal with a comment marker in it)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha(sources=FWD_SOURCES) -> str:
    """Hash of a kernel's code (kernel, PTX helpers, instantiations and the host code that
    sets up its launch; comments and layout excluded): ties a recorded ncu capture to the
    kernel it measured, and a comment edit does not detach it.  The forward's files by
    default; BWD_SOURCES for the backward's kernels."""
    h = hashlib.sha256()
    files = set()
    for pat in sources:
        files.update(glob.glob(os.path.join(ROOT, "tiled_attention_10_gb300", "csrc", pat)))
    for f in sorted(files):
        with open(f, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def use_sustained_peak(total_ms: float, clocks: dict) -> bool:
    """Which measured bf16 GEMM figure the tensor roofline compares with: the sustained one
    (a seconds-long loop under the power cap) when the timed region ran for more than a second
    or under the power cap (sw_power_cap seen by the clock sampler), else the burst one (a
    short loop at full clock)."""
    return total_ms > 1000.0 or "sw_power_cap" in (clocks.get("reasons") or [])


def tensor_peak(peaks, dtype: str, sustained: bool) -> float:
    """Dense tensor peak for the path's dtype: fp8 = 2x the measured bf16 rate
    (the nominal dense ratio, 4.5 vs 2.25 PFLOP/s); f16 = bf16."""
    base = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    return base * (2.0 if dtype == "e4m3" else 1.0)


def recorded_traffic(workload: str, kernel: str = "fa_fwd", sources=FWD_SOURCES):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was
    taken on the current source of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.ncu.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_sha") != kernel_source_sha(sources):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# Clock sampling (nvidia-smi in the background).
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(", ") for ln in self.file.read().splitlines() if ln.strip()]
        self.file.close()
        os.unlink(self.file.name)
        return rows

    @staticmethod
    def summarize(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if len(r) > 2 and num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if len(r) > 3 and num(r[3]) is not None]
        pw = [num(r[4]) for r in rows if len(r) > 4 and num(r[4]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = [name for k, name in enumerate(names)
                   if any(len(r) > 6 + k and r[6 + k].strip() == "Active" for r in rows)]
        loaded = [s for s, p in zip(sm, pw) if p is not None and p > 300] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# Distributed plumbing (barrier and max over ranks only).
# ---------------------------------------------------------------------------
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU baseline: the float64 oracle on the host cores, bounded sample.
# ---------------------------------------------------------------------------
def sample_flops(w, n_heads: int, rows: int) -> float:
    """FLOPs the definition performs for query rows [0, rows) of n_heads
    heads: 4 * D * (keys visible to the row) per row."""
    if w.causal:
        vis = sum(min(i + 1, w.S_kv) for i in range(rows))
    else:
        vis = rows * w.S_kv
    return 4.0 * w.D * vis * n_heads


def oracle_sample(w, x, n_heads: int, rows: int, threads: int = 0) -> float:
    """Oracle over query rows [0, rows) of the first n_heads (b, h) heads;
    returns seconds."""
    import oracle
    import torch
    heads = []
    g = w.H // w.kv_heads
    for bh in range(n_heads):
        b, h = divmod(bh, w.H)
        if w.layout == "BNSD":
            heads.append((x.q[b, h, :rows], x.k[b, h // g], x.v[b, h // g]))
        else:
            heads.append((x.q[b, :rows, h], x.k[b, :, h // g], x.v[b, :, h // g]))
    q = torch.stack([t[0] for t in heads]).unsqueeze(0).cpu()
    k = torch.stack([t[1] for t in heads]).unsqueeze(0).cpu()
    v = torch.stack([t[2] for t in heads]).unsqueeze(0).cpu()
    t0 = time.perf_counter()
    oracle.attention_full(q, k, v, dtype=w.dtype, layout="BNSD", B=1, H=n_heads, S_q=rows,
                          S_kv=w.S_kv, D=w.D, scale=w.softmax_scale, causal=w.causal,
                          descale=x.descale, threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(w, x, budget_s: float = 12.0):
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    rows = min(w.S_q, 512)
    t1 = oracle_sample(w, x, 1, rows)
    n = int(max(1, min(w.B * w.H, budget_s / max(t1, 1e-3))))
    t = oracle_sample(w, x, n, rows) if n > 1 else t1
    return {"value": round(sample_flops(w, n, rows) / t / 1e12, 6), "unit": "TFLOP/s",
            "cores": cores, "kind": "oracle",
            "sample": f"query rows [0, {rows}) of {n} of {w.B * w.H} (batch, head) pairs, "
                      f"float64, {t:.1f} s"}


def oracle_bwd_head(w, x, do, b: int = 0, hk: int = 0) -> float:
    """Backward oracle for one key/value head (all query heads that read it);
    returns seconds."""
    from oracle import backward as ob
    t0 = time.perf_counter()
    ob.attention_bwd(x.q, x.k, x.v, do, dtype=w.dtype, layout=w.layout, B=w.B, H=w.H,
                     S_q=w.S_q, S_kv=w.S_kv, D=w.D, scale=w.softmax_scale, causal=w.causal,
                     H_kv=w.kv_heads, kv_heads=[(b, hk)])
    return time.perf_counter() - t0


def bwd_sample_flops(w) -> float:
    """Nominal backward FLOPs of one key/value head's query heads."""
    return w.flops / (w.B * w.kv_heads)


def cpu_baseline_bwd(w, x, do):
    import oracle
    oracle.build()
    t = oracle_bwd_head(w, x, do)
    return {"value": round(bwd_sample_flops(w) / t / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"one (batch, key/value head) of {w.B * w.kv_heads}: {w.H // w.kv_heads} "
                      f"query head(s) x {w.S_q} x {w.S_kv}, float64 numpy, {t:.1f} s"}


def visible_pairs(w) -> int:
    """(query, key) pairs the mask leaves visible over the whole workload:
    one exponential each in the softmax (top-left causal: row i sees keys
    0..min(i, S_kv - 1))."""
    if not w.causal:
        per_head = w.S_q * w.S_kv
    else:
        n = min(w.S_q, w.S_kv)            # rows 0..n-1 see i + 1 keys
        per_head = n * (n + 1) // 2 + max(0, w.S_q - n) * w.S_kv
    return w.B * w.H * per_head


def secondary_ceilings(pairs: int, launch_s: float, sms: int, sm_mhz: float, clock_src: str):
    """The softmax's own ceilings beside the tensor roofline: the MUFU unit's
    exponentials (one ex2 per visible pair, 32 per clock per SM, measured with
    a microbenchmark) and the FP32 pipe's softmax arithmetic (three operations
    per visible pair -- the scale-and-subtract FMA, the max and the row-sum add
    -- at 128 per clock per SM)."""
    hz = sm_mhz * 1e6
    out = {}
    for name, per_pair, per_clk in (("mufu_ex2", 1, 32), ("fp32_softmax", 3, 128)):
        ops = per_pair * pairs
        peak = per_clk * sms * hz
        out[name] = {"ops_per_launch": ops, "achieved_per_s": round(ops / launch_s, 1),
                     "peak_per_s": round(peak, 1), "frac": round(ops / launch_s / peak, 4),
                     "peak_source": f"{per_clk} per clock per SM x {sms} SMs x {sm_mhz:.0f} MHz "
                                    f"({clock_src})"}
    return out


def timing_summary(per_launch_ms, flops=None):
    """Mean, median and min of the per-call CUDA-event times (and the TFLOP/s
    each gives)."""
    t = {"ms_mean": round(statistics.mean(per_launch_ms), 5),
         "ms_median": round(statistics.median(per_launch_ms), 5),
         "ms_min": round(min(per_launch_ms), 5),
         "how": "a second pass of as many calls right after the timed region, a CUDA event "
                "on the launching stream between consecutive calls"}
    if flops:
        for k in ("mean", "median", "min"):
            t[f"tflops_{k}"] = round(flops / (t[f"ms_{k}"] * 1e-3) / 1e12, 2)
    return t


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def run_oracle_full(args, w, world, rank):
    """The float64 oracle timed on the whole workload on the host cores (every
    row); for a workload too large for that, on seeded sample rows with the
    full time extrapolated by FLOPs (and labelled so).  One JSON line."""
    if rank != 0:
        return 0
    import oracle
    import torch
    from tiled_attention_10_gb300.inputs import make_inputs, sample_rows
    oracle.build()
    cores = oracle.max_threads()
    full = w.B * w.H * w.S_q * w.S_kv <= (1 << 34)
    line = {"oracle_full": w.name, "cores": cores, "cpu": cpu_model(), "dtype": "f64",
            "nominal_flops": w.flops}
    if full:
        x = make_inputs(w)
        t0 = time.perf_counter()
        oracle.attention_full(x.q, x.k, x.v, dtype=w.dtype, layout=w.layout, B=w.B, H=w.H,
                              S_q=w.S_q, S_kv=w.S_kv, D=w.D, scale=w.softmax_scale,
                              causal=w.causal, descale=x.descale, H_kv=w.kv_heads)
        t = time.perf_counter() - t0
        line.update({"seconds": round(t, 3), "gflops": round(w.flops / t / 1e9, 3),
                     "scope": "every row of every head", "extrapolated": False})
    else:
        # Every row of one (batch, head) pair -- the same shape per head as the
        # whole workload -- timed on all cores, then scaled by FLOPs to the
        # B*H pairs (labelled as an extrapolation); plus the 64 seeded sample
        # rows the parity test checks, one oracle call each.
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        x = make_inputs(w, device=dev)
        if w.layout == "BNSD":
            qh, kh, vh = x.q[:1, :1].cpu(), x.k[:1, :1].cpu(), x.v[:1, :1].cpu()
        else:
            qh, kh, vh = (x.q[:1, :, :1].cpu(), x.k[:1, :, :1].cpu(), x.v[:1, :, :1].cpu())
        t0 = time.perf_counter()
        oracle.attention_full(qh, kh, vh, dtype=w.dtype, layout=w.layout, B=1, H=1, S_q=w.S_q,
                              S_kv=w.S_kv, D=w.D, scale=w.softmax_scale, causal=w.causal,
                              descale=x.descale)
        t_head = time.perf_counter() - t0
        head_flops = w.flops / (w.B * w.H)
        rows = [tuple(int(v) for v in r) for r in sample_rows(w, 64, seed=0)]
        g = w.H // w.kv_heads
        spent = 0.0
        for (b, h, i) in rows:
            hk = h // g
            if w.layout == "BNSD":
                qr, kr, vr = x.q[b, h].cpu(), x.k[b, hk].cpu(), x.v[b, hk].cpu()
            else:
                qr, kr, vr = x.q[b, :, h].cpu(), x.k[b, :, hk].cpu(), x.v[b, :, hk].cpu()
            t0 = time.perf_counter()
            oracle.attention_rows(qr, kr, vr, dtype=w.dtype, layout="BNSD", B=1, H=1, S_q=w.S_q,
                                  S_kv=w.S_kv, D=w.D, scale=w.softmax_scale, causal=w.causal,
                                  rows=[(0, 0, i)], descale=x.descale)
            spent += time.perf_counter() - t0
        line.update({"seconds_one_head": round(t_head, 3),
                     "gflops_one_head": round(head_flops / t_head / 1e9, 3),
                     "seconds": round(t_head * w.B * w.H, 1), "extrapolated": True,
                     "scope": f"extrapolated: every row of (batch 0, head 0) timed, times the "
                              f"{w.B * w.H} (batch, head) pairs",
                     "sample_rows": len(rows), "seconds_sample_rows": round(spent, 3),
                     "seconds_per_sample_row": round(spent / len(rows), 4)})
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Arms.
# ---------------------------------------------------------------------------
def run_reference(args, w, world, rank):
    """The reference arm: the float64 oracle on the host cores, one bounded
    sample of the workload (query rows of one head) per step."""
    if rank != 0:
        return 0
    import oracle
    from tiled_attention_10_gb300.inputs import make_dout, make_inputs
    oracle.build()
    if w.bwd:
        one = type(w)(**{**w.__dict__, "B": 1, "H": w.H // w.kv_heads, "H_kv": 1})
        x, do = make_inputs(one), make_dout(one)
        for _ in range(args.warmup):
            oracle_bwd_head(one, x, do)
        times = [oracle_bwd_head(one, x, do) for _ in range(args.steps)]
        t = sum(times) / len(times)
        val = bwd_sample_flops(one) / t / 1e12
        sample = (f"backward of one (batch, key/value head) per step: {one.H} query head(s) x "
                  f"{w.S_q} x {w.S_kv}, float64")
        cores = oracle.max_threads()
        line = {"impl": "reference", "metric": "attention bwd TFLOP/s", "value": round(val, 6),
                "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {**w.describe(), "sample_per_step": sample},
                "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": cores,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0
    one = type(w)(**{**w.__dict__, "B": 1, "H": 1, "H_kv": None})
    x = make_inputs(one)
    cores = oracle.max_threads()
    rows = min(w.S_q, 256)
    for _ in range(args.warmup):
        oracle_sample(one, x, 1, rows)
    times = [oracle_sample(one, x, 1, rows) for _ in range(args.steps)]
    t = sum(times) / len(times)
    val = sample_flops(one, 1, rows) / t / 1e12
    sample = f"query rows [0, {rows}) of one (batch, head) pair per step, float64"
    line = {"impl": "reference", "metric": "attention fwd TFLOP/s", "value": round(val, 6),
            "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**w.describe(), "sample_per_step": sample},
            "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


E2E_STREAMED = ("streamed: each step's inputs host->device on one copy stream and its results "
                "device->host on another, through one of two device buffer sets, so the copies "
                "of neighbouring steps overlap a step's compute; every step copies all of its "
                "inputs in and all of its results out inside the timed region")
E2E_SERIAL = ("serial: each step copies its inputs host->device, computes and copies its results "
              "device->host on one stream (steps this small are bound by the host's per-call "
              "overhead, which streaming only adds to)")
E2E_STREAM_MIN_BYTES = 16 << 20   # stream the steps whose inputs are at least this large


def e2e_ms_per_step(torch, stream, host_in, dev_in, run, dev_out, host_out, steps, world):
    """End to end through the public call with pinned host buffers, fed the way a caller
    streams batches: E2E_STREAMED when a step's inputs are at least E2E_STREAM_MIN_BYTES,
    else E2E_SERIAL.  dev_in / dev_out: two lists of device tensors (one per buffer set);
    run(b) computes from dev_in[b] into dev_out[b] on `stream`.  Returns (mean ms per step
    over `steps` steps by CUDA events, max over ranks; the description of the scheme)."""
    streamed = sum(t.numel() * t.element_size() for t in host_in) >= E2E_STREAM_MIN_BYTES
    h2d, d2h = (torch.cuda.Stream(), torch.cuda.Stream()) if streamed else (stream, stream)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    out_home = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def one(i):
        if not streamed:
            for d_, h_ in zip(dev_in[0], host_in):
                d_.copy_(h_, non_blocking=True)
            run(0)
            for h_, d_ in zip(host_out, dev_out[0]):
                h_.copy_(d_, non_blocking=True)
            return
        b = i % 2
        with torch.cuda.stream(h2d):
            if used[b]:
                h2d.wait_event(computed[b])        # step i-2 has read this set's inputs
            for d_, h_ in zip(dev_in[b], host_in):
                d_.copy_(h_, non_blocking=True)
            in_ready[b].record(h2d)
        stream.wait_event(in_ready[b])
        if used[b]:
            stream.wait_event(out_home[b])         # step i-2's results have left this set
        run(b)
        computed[b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(computed[b])
            for h_, d_ in zip(host_out, dev_out[b]):
                h_.copy_(d_, non_blocking=True)
            out_home[b].record(d2h)
        used[b] = True

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    if streamed:
        h2d.wait_stream(stream)                    # no copy starts before e0
    for i in range(steps):
        one(i)
    if streamed:
        stream.wait_stream(d2h)
    e1.record(stream)
    torch.cuda.synchronize()
    return (max_over_ranks(e0.elapsed_time(e1) / steps, world),
            E2E_STREAMED if streamed else E2E_SERIAL)


def timed_steps(torch, stream, step, steps, world):
    """The timed region: `steps` calls between two CUDA events on the launching
    stream, bracketed by a barrier and a synchronize on both sides; returns its
    milliseconds.  Then, outside it, the same number of calls each between its
    own pair of events (events between calls add a little per call, which
    matters for calls of a few microseconds): the per-call list for the median
    and minimum."""
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = e0.elapsed_time(e1)
    timed_steps.host_us = None
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    # Host time to issue one call (argument checks, tensor maps, launch), by
    # the wall clock over a burst of calls that the device has not caught up
    # with: when it is below the per-call device time, the device sets the pace.
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    timed_steps.host_us = (time.perf_counter() - t0) / steps * 1e6
    torch.cuda.synchronize()
    return total_ms, [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]


def run_ours(args, w, world, rank, local):
    import torch
    from tiled_attention_10_gb300 import binding
    from tiled_attention_10_gb300.inputs import OUT_DTYPE, make_inputs, shape_of

    binding.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    if world > 1:   # each rank: its own independent shard of B*H heads (weak scaling)
        w = type(w)(**{**w.__dict__, "seed": w.seed + 1000 * rank})
    x = make_inputs(w, device=dev)
    q, k, v = x.q, x.k, x.v
    o = torch.empty(shape_of(w.layout, w.B, w.H, w.S_q, w.D), dtype=OUT_DTYPE[w.dtype], device=dev)
    lse = torch.empty(w.B, w.H, w.S_q, dtype=torch.float32, device=dev)
    ds = [None, None, None]
    if w.dtype == "e4m3":
        dst = [torch.tensor([d], dtype=torch.float32, device=dev) for d in x.descale]
        ds = [t.data_ptr() for t in dst]
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    n_splits, ws, ws_bytes = 1, None, 0
    if w.split:   # split-KV: plan once, workspace allocated outside the timed region
        st, n_splits, ws_bytes = binding.fa_fwd_splitkv_plan(w.B, w.H, w.S_q, w.S_kv, w.D)
        if st != 0:
            raise RuntimeError("fa_fwd_splitkv_plan failed")
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    launches_per_step = 2 if n_splits > 1 else 1

    def step(qq=q, kk=k, vv=v, oo=o, ll=lse):
        if w.split:
            st = binding.fa_fwd_splitkv(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), oo.data_ptr(),
                                        ll.data_ptr(), w.B, w.H, w.kv_heads, w.S_q, w.S_kv, w.D,
                                        w.softmax_scale, w.layout, w.causal, w.dtype, ds[0],
                                        ds[1], ds[2], n_splits, ws.data_ptr(), ws_bytes, sp)
        else:
            st = binding.fa_fwd_gqa(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), oo.data_ptr(),
                                    ll.data_ptr(), w.B, w.H, w.kv_heads, w.S_q, w.S_kv, w.D,
                                    w.softmax_scale, w.layout, w.causal, w.dtype, ds[0], ds[1],
                                    ds[2], sp)
        if st != 0:
            raise RuntimeError(f"fa_fwd: {binding.fa_status_string(st)}")

    sampler = ClockSampler(local)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if binding.fa_last_device_error(sp) != 0:
        raise RuntimeError("device-side error during warm-up")

    total_ms, per_launch = timed_steps(torch, stream, step, args.steps, world)
    clocks = ClockSampler.summarize(sampler.stop())
    ms = total_ms / args.steps
    ms_max = max_over_ranks(ms, world)
    if binding.fa_last_device_error(sp) != 0:
        raise RuntimeError("device-side error during the timed steps")

    # End to end through the public call: pinned host inputs in, O and lse out.
    host_in = [t.cpu().pin_memory() for t in (q, k, v)]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse)]
    dev_in = [[torch.empty_like(t) for t in (q, k, v)] for _ in range(2)]
    dev_out = [[o, lse], [torch.empty_like(o), torch.empty_like(lse)]]
    e2e_ms, e2e_how = e2e_ms_per_step(torch, stream, host_in, dev_in,
                             lambda b: step(*dev_in[b], *dev_out[b]), dev_out, host_out,
                             max(1, min(args.steps, 50)), world)
    h2d = (q.numel() * q.element_size()) + (k.numel() * k.element_size()) + (v.numel() * v.element_size())
    d2h = o.numel() * o.element_size() + lse.numel() * 4

    if rank != 0:
        return 0
    flops = w.flops
    value = world * flops / (ms_max * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    sustained = use_sustained_peak(total_ms, clocks)
    peak = tensor_peak(peaks, w.dtype, sustained)
    launch_ms = ms
    achieved = flops / (launch_ms * 1e-3) / 1e12
    in_bytes = h2d
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clk, clk_src = ((clocks["sm_mhz"], "median SM clock sampled during the timed calls")
                    if clocks.get("sm_mhz") else (peaks.get("sm_max_mhz", 2070.0), "maximum SM clock"))
    line = {
        "metric": "attention fwd TFLOP/s", "value": round(value, 3), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {**w.describe(),
                   "l2": ("no flush: inputs (Q+K+V) exceed the 129 MB L2" if in_bytes > (129 << 20)
                          else "no flush: inputs fit in L2 (launch-bound workload)"),
                   "parallelism": f"{world} independent shard(s) of B*H, one per GPU",
                   **({"n_splits": n_splits} if w.split else {})},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     **({"frac_of_burst": round(achieved / tensor_peak(peaks, w.dtype, False), 4)}
                        if sustained else {}),
                     "traffic": recorded_traffic(w.name),
                     "peak_source": f"{peak_src} {'sustained' if sustained else 'burst'} bf16 GEMM"
                                    f"{' x2 (fp8 nominal ratio)' if w.dtype == 'e4m3' else ''}",
                     "secondary": secondary_ceilings(visible_pairs(w), launch_ms * 1e-3, sms, clk,
                                                     clk_src)},
        "timing": {**timing_summary(per_launch, flops),
                   "host_us_per_call": round(timed_steps.host_us, 2)},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "how": e2e_how},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, x)
    print(json.dumps(line), flush=True)
    return 0


def run_ours_bwd(args, w, world, rank, local):
    """Backward workloads: one step = one fa_bwd call (three launches: row
    statistics, dQ kernel, dK/dV kernel) with Q, K, V, O, dO, lse resident."""
    import torch
    from tiled_attention_10_gb300 import binding
    from tiled_attention_10_gb300.inputs import make_dout, make_inputs

    binding.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    if world > 1:
        w = type(w)(**{**w.__dict__, "seed": w.seed + 1000 * rank})
    x = make_inputs(w, device=dev)
    q, k, v = x.q, x.k, x.v
    do = make_dout(w, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.S_q, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    st = binding.fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            w.B, w.H, w.kv_heads, w.S_q, w.S_kv, w.D, w.softmax_scale, w.layout,
                            w.causal, w.dtype, None, None, None, sp)
    if st != 0:
        raise RuntimeError(f"fa_fwd: {binding.fa_status_string(st)}")
    st, ws_bytes = binding.fa_bwd_workspace_size(w.B, w.H, w.S_q)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def step(qq=q, kk=k, vv=v, oo=o, dd=do, ll=lse, gq=dq, gk=dk, gv=dv):
        st = binding.fa_bwd(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), oo.data_ptr(),
                            dd.data_ptr(), ll.data_ptr(), gq.data_ptr(), gk.data_ptr(),
                            gv.data_ptr(), w.B, w.H, w.kv_heads, w.S_q, w.S_kv, w.D,
                            w.softmax_scale, w.layout, w.causal, w.dtype, ws.data_ptr(), ws_bytes,
                            sp)
        if st != 0:
            raise RuntimeError(f"fa_bwd: {binding.fa_status_string(st)}")

    sampler = ClockSampler(local)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if binding.fa_last_device_error(sp) != 0:
        raise RuntimeError("device-side error during warm-up")
    total_ms, per_step = timed_steps(torch, stream, step, args.steps, world)
    clocks = ClockSampler.summarize(sampler.stop())
    ms_max = max_over_ranks(total_ms / args.steps, world)
    if binding.fa_last_device_error(sp) != 0:
        raise RuntimeError("device-side error during the timed steps")

    # End to end: pinned host Q, K, V, O, dO, lse in; dQ, dK, dV out.
    ins = (q, k, v, o, do, lse)
    host_in = [t.cpu().pin_memory() for t in ins]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
    dev_in = [[torch.empty_like(t) for t in ins] for _ in range(2)]
    dev_out = [[dq, dk, dv], [torch.empty_like(t) for t in (dq, dk, dv)]]
    e2e_ms, e2e_how = e2e_ms_per_step(torch, stream, host_in, dev_in,
                             lambda b: step(*dev_in[b], *dev_out[b]), dev_out, host_out,
                             max(1, min(args.steps, 30)), world)
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in (dq, dk, dv))
    if rank != 0:
        return 0
    flops = w.flops
    peaks, peak_src = load_peaks()
    sustained = use_sustained_peak(total_ms, clocks)
    peak = tensor_peak(peaks, w.dtype, sustained)
    step_ms = total_ms / args.steps
    achieved = flops / (step_ms * 1e-3) / 1e12
    # Products the tensor cores actually run per step: the dQ kernel
    # recomputes S and dP, so 7 forward-sized products against the 5 counted.
    executed = flops * 7.0 / 5.0 / (step_ms * 1e-3) / 1e12
    line = {
        "metric": "attention bwd TFLOP/s", "value": round(world * flops / (ms_max * 1e-3) / 1e12, 3),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {**w.describe(),
                   "l2": "no flush: inputs (Q, K, V, O, dO) exceed the 129 MB L2",
                   "parallelism": f"{world} independent shard(s) of B*H, one per GPU",
                   "flops": "2.5 x the forward's 4*B*H*S_q*S_kv*D (halved when causal)"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     **({"frac_of_burst": round(achieved / tensor_peak(peaks, w.dtype, False), 4)}
                        if sustained else {}),
                     "traffic": None,
                     "traffic_by_kernel": {k: recorded_traffic(w.name, k, BWD_SOURCES)
                                           for k in ("fa_bwd_dq", "fa_bwd_dkdv")},
                     "scope": "whole fa_bwd step (row statistics + dQ + dK/dV kernels, CUDA "
                              "events around each call)",
                     "executed_frac": round(executed / peak, 4),
                     "peak_source": f"{peak_src} {'sustained' if sustained else 'burst'} bf16 GEMM"},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "how": e2e_how},
        "timing": timing_summary(per_step, flops),
        "gpu_launches": args.steps * 3,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_bwd(w, make_inputs(w), make_dout(w))
    print(json.dumps(line), flush=True)
    return 0


def packed_oracle_sample(w, x):
    """Oracle on the packed workload's cheapest sequence (all heads): returns
    (seconds, FLOPs of that sequence, description)."""
    from oracle import varlen as ov
    import numpy as np
    cost = [sq * sk for sq, sk in zip(w.seq_q, w.seq_k)]
    s = int(np.argmin(cost))
    cu_q = x.cu_q.cpu().numpy()
    t0 = time.perf_counter()
    if w.page_size:
        ov.attention_paged(x.q.cpu(), x.k.cpu(), x.v.cpu(), cu_q=cu_q,
                           seqused_k=x.seqused_k.cpu().numpy(), block_table=x.block_table.cpu().numpy(),
                           page_size=w.page_size, H=w.H, H_kv=w.H_kv, D=w.D, scale=w.softmax_scale,
                           causal_mode=w.causal, dtype=w.dtype, descale=x.descale, seqs=[s])
    else:
        ov.attention_varlen(x.q.cpu(), x.k.cpu(), x.v.cpu(), cu_q=cu_q, cu_k=x.cu_k.cpu().numpy(),
                            H=w.H, H_kv=w.H_kv, D=w.D, scale=w.softmax_scale, causal_mode=w.causal,
                            dtype=w.dtype, descale=x.descale, seqs=[s])
    t = time.perf_counter() - t0
    one = type(w)(**{**w.__dict__, "seq_q": (w.seq_q[s],), "seq_k": (w.seq_k[s],)})
    return t, one, f"sequence {s} ({w.seq_q[s]} x {w.seq_k[s]}), all {w.H} heads, float64 numpy"


def run_reference_packed(args, w, world, rank):
    """Reference arm for packed workloads: the float64 oracle on the cheapest
    sequence of the batch per step."""
    if rank != 0:
        return 0
    import oracle
    from tiled_attention_10_gb300.inputs import make_packed_inputs
    x = make_packed_inputs(w)
    for _ in range(args.warmup):
        packed_oracle_sample(w, x)
    runs = [packed_oracle_sample(w, x) for _ in range(args.steps)]
    t = sum(r[0] for r in runs) / len(runs)
    one, sample = runs[0][1], runs[0][2]
    if w.decode:
        metric, unit, val = "attention decode GB/s", "GB/s", one.kv_bytes / t / 1e9
    else:
        metric, unit, val = "attention fwd TFLOP/s", "TFLOP/s", one.flops / t / 1e12
    line = {"impl": "reference", "metric": metric, "value": round(val, 6), "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**w.describe(), "sample_per_step": sample},
            "cpu_baseline": {"value": round(val, 6), "unit": unit, "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 6), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours_packed(args, w, world, rank, local):
    """Packed workloads: one step = one fa_fwd_varlen / fa_fwd_paged call."""
    import torch
    from tiled_attention_10_gb300 import binding
    from tiled_attention_10_gb300.inputs import OUT_DTYPE, make_packed_inputs

    binding.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    if world > 1:
        w = type(w)(**{**w.__dict__, "seed": w.seed + 1000 * rank})
    x = make_packed_inputs(w, device=dev)
    tq = sum(w.seq_q)
    o = torch.empty(tq, w.H, w.D, dtype=OUT_DTYPE[w.dtype], device=dev)
    lse = torch.empty(w.H, tq, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    ds = [None, None, None]
    if w.dtype == "e4m3":
        dst = [torch.tensor([d], dtype=torch.float32, device=dev) for d in x.descale]
        ds = [t.data_ptr() for t in dst]

    # paged split: n_splits given, or (0) planned from the host-known sizes;
    # the workspace is allocated outside the timed region
    ws, ws_bytes, n_splits = None, 0, w.n_splits
    use_split = bool(w.page_size) and n_splits != 1
    if use_split:
        if n_splits == 0:
            st, n_splits, _ = binding.fa_fwd_paged_split_plan(len(w.seq_q), tq, max(w.seq_q),
                                                              sum(w.seq_k), max(w.seq_k), w.H,
                                                              w.H_kv, w.D)
            if st != 0:
                raise RuntimeError(f"paged split plan: {binding.fa_status_string(st)}")
        st, ws_bytes = binding.fa_fwd_paged_split_workspace_size(w.H, tq, w.D, n_splits,
                                                                 len(w.seq_q))
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    # launches per step: paged split = sequence-order pre-pass (up to 16384
    # sequences), forward, and the merge when the keys are split
    launches_per_step = (1 + (len(w.seq_q) <= 16384) + (n_splits > 1)) if use_split else 1

    def step(qq=x.q, kk=x.k, vv=x.v, oo=o, ll=lse):
        if use_split:
            st = binding.fa_fwd_paged_split(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(),
                                            oo.data_ptr(), ll.data_ptr(), x.cu_q.data_ptr(),
                                            x.seqused_k.data_ptr(), x.block_table.data_ptr(),
                                            len(w.seq_q), x.block_table.shape[1], w.page_size,
                                            kk.shape[0], tq, max(w.seq_q), w.H, w.H_kv, w.D,
                                            w.softmax_scale, w.causal, w.dtype, *ds, n_splits,
                                            ws.data_ptr(), ws_bytes, sp)
        elif w.page_size:
            st = binding.fa_fwd_paged(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), oo.data_ptr(),
                                      ll.data_ptr(), x.cu_q.data_ptr(), x.seqused_k.data_ptr(),
                                      x.block_table.data_ptr(), len(w.seq_q), x.block_table.shape[1],
                                      w.page_size, kk.shape[0], tq, max(w.seq_q), w.H, w.H_kv, w.D,
                                      w.softmax_scale, w.causal, w.dtype, *ds, sp)
        else:
            st = binding.fa_fwd_varlen(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), oo.data_ptr(),
                                       ll.data_ptr(), x.cu_q.data_ptr(), x.cu_k.data_ptr(),
                                       len(w.seq_q), tq, sum(w.seq_k), max(w.seq_q), w.H, w.H_kv,
                                       w.D, w.softmax_scale, w.causal, w.dtype, *ds, sp)
        if st != 0:
            raise RuntimeError(f"packed forward: {binding.fa_status_string(st)}")

    sampler = ClockSampler(local)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if binding.fa_last_device_error(sp) != 0:
        raise RuntimeError("device-side error during warm-up")
    total_ms, per_launch = timed_steps(torch, stream, step, args.steps, world)
    clocks = ClockSampler.summarize(sampler.stop())
    ms_max = max_over_ranks(total_ms / args.steps, world)
    if binding.fa_last_device_error(sp) != 0:
        raise RuntimeError("device-side error during the timed steps")

    # End to end: pinned host Q and K / V (or caches) in, O and lse out.
    host_in = [t.cpu().pin_memory() for t in (x.q, x.k, x.v)]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse)]
    dev_in = [[torch.empty_like(t) for t in (x.q, x.k, x.v)] for _ in range(2)]
    dev_out = [[o, lse], [torch.empty_like(o), torch.empty_like(lse)]]
    e2e_ms, e2e_how = e2e_ms_per_step(torch, stream, host_in, dev_in,
                             lambda b: step(*dev_in[b], *dev_out[b]), dev_out, host_out,
                             max(1, min(args.steps, 20)), world)
    h2d = sum(t.numel() * t.element_size() for t in (x.q, x.k, x.v))
    d2h = o.numel() * o.element_size() + lse.numel() * 4
    if rank != 0:
        return 0
    peaks, peak_src = load_peaks()
    launch_ms = total_ms / args.steps
    q_bytes = x.q.numel() * x.q.element_size()
    algo_bytes = w.kv_bytes + q_bytes + d2h       # K / V read once, Q read, O and lse written
    if w.decode:
        metric, unit = "attention decode GB/s", "GB/s"
        value = world * algo_bytes / (ms_max * 1e-3) / 1e9
        achieved = algo_bytes / (launch_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": None,
                "algorithmic_bytes": algo_bytes,
                "peak_source": f"{peak_src} HBM copy bandwidth"}
        e2e_val = world * algo_bytes / (e2e_ms * 1e-3) / 1e9
    else:
        metric, unit = "attention fwd TFLOP/s", "TFLOP/s"
        value = world * w.flops / (ms_max * 1e-3) / 1e12
        achieved = w.flops / (launch_ms * 1e-3) / 1e12
        sustained = use_sustained_peak(total_ms, clocks)
        peak = tensor_peak(peaks, w.dtype, sustained)
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                **({"frac_of_burst": round(achieved / tensor_peak(peaks, w.dtype, False), 4)}
                   if sustained else {}),
                "traffic": None,
                "peak_source": f"{peak_src} {'sustained' if sustained else 'burst'} bf16 GEMM"}
        e2e_val = world * w.flops / (e2e_ms * 1e-3) / 1e12
    line = {
        "metric": metric, "value": round(value, 3), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {**w.describe(),
                   "flops": "4*D*H per visible (query, key) pair",
                   "l2": ("no flush: K/V exceed the 129 MB L2" if w.kv_bytes > (129 << 20)
                          else "no flush: inputs fit in L2"),
                   **({"n_splits": n_splits} if use_split else {}),
                   "parallelism": f"{world} independent shard(s), one per GPU"},
        "roofline": roof,
        "e2e": {"value": round(e2e_val, 3), "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "how": e2e_how},
        "timing": timing_summary(per_launch, None if w.decode else w.flops),
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        t, one, sample = packed_oracle_sample(w, make_packed_inputs(w))
        val = (one.flops / t / 1e12) if not w.decode else (one.kv_bytes / t / 1e9)
        line["cpu_baseline"] = {"value": round(val, 6), "unit": unit,
                                "cores": oracle.max_threads(), "kind": "oracle",
                                "sample": f"{sample}, {t:.2f} s"}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description="FlashAttention forward benchmark (libfa_b200)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-full", action="store_true",
                    help="time the float64 oracle on the whole workload (host cores) and exit")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from tiled_attention_10_gb300.inputs import ALL_WORKLOADS, HEADLINE, PACKED_WORKLOADS
    w = {**ALL_WORKLOADS, **PACKED_WORKLOADS}[args.workload or HEADLINE]
    world, rank, local = dist_setup()
    try:
        if args.oracle_full:
            return run_oracle_full(args, w, world, rank)
        if hasattr(w, "seq_q"):
            if args.impl == "reference":
                return run_reference_packed(args, w, world, rank)
            return run_ours_packed(args, w, world, rank, local)
        if args.impl == "reference":
            return run_reference(args, w, world, rank)
        if w.bwd:
            return run_ours_bwd(args, w, world, rank, local)
        return run_ours(args, w, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
