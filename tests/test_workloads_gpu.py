"""The five measured workloads at full size, in the launch configuration the
benchmark times, against the float64 oracle.

  fp16_1x8x512x64                  every row
  bf16_bsnd_causal_2x16x4097x64    every row (NaN-poisoned memory past the tail)
  bf16_4x32x4096x128               sampled rows (corners, tile edges, random)
  fp8_causal_1x32x8192x128         every row of two heads + sampled rows
  bf16_causal_16x64x16384x128      64 seeded (b, h, row) samples; each tensor
                                   holds 2^31 elements (> 4 GB)
Plus, at every size, properties that need no oracle: no NaN/Inf anywhere in
O or lse, canaries after the outputs intact.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_10_gb300.inputs import EXTRA_WORKLOADS, WORKLOADS, make_inputs, sample_rows
from tests.gpu_helpers import TOL_LSE, TOL_O, Run, check, compare_full, sampled_rows_check, to_device

pytestmark = pytest.mark.gpu


def _whole_output_finite(r: Run) -> bool:
    return bool(torch.isfinite(r.o.float()).all()) and bool(torch.isfinite(r.lse).all())


@pytest.mark.parametrize("name", ["fp16_1x8x512x64", "bf16_bsnd_causal_2x16x4097x64"])
def test_workload_every_row(name, cuda_lib):
    w = WORKLOADS[name]
    x = make_inputs(w)
    q, k, v = to_device(x)
    r = Run(w, q, k, v, descale=x.descale)
    torch.cuda.synchronize()
    eo, el, og, lg = compare_full(w, r, x)
    check(w, r, eo, el, og, lg)
    print(f"{name}: max|dO|={eo:.3g} max|dlse|={el:.3g}")


def _edge_rows(w, n_random, seed=0):
    rows = [tuple(int(v) for v in t) for t in sample_rows(w, n_random, seed)]
    S = w.S_q
    for i in (1, 127, 128, 129, 255, 256, S // 2, S - 129, S - 128, S - 2, S - 1):
        if 0 <= i < S:
            rows.append((w.B - 1, 0, i))
            rows.append((0, w.H - 1, i))
    return sorted(set(rows))


def test_workload_headline_bf16_sampled(cuda_lib):
    w = WORKLOADS["bf16_4x32x4096x128"]
    x = make_inputs(w, device="cuda")
    r = Run(w, x.q, x.k, x.v)
    torch.cuda.synchronize()
    assert r.status == 0 and r.device_status == 0 and r.guards_intact()
    assert _whole_output_finite(r)
    eo, el = sampled_rows_check(w, r, x.q, x.k, x.v, x.descale, _edge_rows(w, 200))
    assert eo <= TOL_O[w.dtype] and el <= TOL_LSE, (eo, el)
    print(f"headline: max|dO|={eo:.3g} max|dlse|={el:.3g}")


def test_workload_fp8_causal(cuda_lib):
    w = WORKLOADS["fp8_causal_1x32x8192x128"]
    x = make_inputs(w, device="cuda")
    r = Run(w, x.q, x.k, x.v, descale=x.descale)
    torch.cuda.synchronize()
    assert r.status == 0 and r.device_status == 0 and r.guards_intact()
    assert _whole_output_finite(r)
    # every row of two heads (the short causal rows are where P quantisation bites)
    for h in (0, w.H - 1):
        O, lse = oracle.attention_full(x.q[:, h:h + 1].cpu(), x.k[:, h:h + 1].cpu(),
                                       x.v[:, h:h + 1].cpu(), dtype="e4m3", layout="BNSD", B=1,
                                       H=1, S_q=w.S_q, S_kv=w.S_kv, D=w.D,
                                       scale=w.softmax_scale, causal=True, descale=x.descale)
        og = r.o[:, h:h + 1].float().cpu().double().numpy()
        lg = r.lse[:, h:h + 1].cpu().double().numpy()
        eo, el = float(np.abs(og - O).max()), float(np.abs(lg - lse).max())
        print(f"fp8 head {h}: max|dO|={eo:.3g} max|dlse|={el:.3g}")
        assert eo <= TOL_O["e4m3"] and el <= TOL_LSE, (h, eo, el)
    eo, el = sampled_rows_check(w, r, x.q, x.k, x.v, x.descale, _edge_rows(w, 64, seed=1))
    assert eo <= TOL_O["e4m3"] and el <= TOL_LSE, (eo, el)


@pytest.mark.slow
def test_workload_over_4gb_causal(cuda_lib):
    w = WORKLOADS["bf16_causal_16x64x16384x128"]
    assert w.B * w.H * w.S_q * w.D == 2 ** 31          # 4.29 GB per bf16 tensor
    x = make_inputs(w, device="cuda")
    r = Run(w, x.q, x.k, x.v)
    torch.cuda.synchronize()
    assert r.status == 0 and r.device_status == 0 and r.guards_intact()
    assert _whole_output_finite(r)
    rows = [tuple(int(v) for v in t) for t in sample_rows(w, 64, seed=0)]
    eo, el = sampled_rows_check(w, r, x.q, x.k, x.v, x.descale, rows)
    print(f"over-4GB: max|dO|={eo:.3g} max|dlse|={el:.3g} on {len(rows)} rows")
    assert eo <= TOL_O[w.dtype] and el <= TOL_LSE, (eo, el)
    # the last head's last rows live beyond byte offset 2^32 of every tensor
    tail = [(w.B - 1, w.H - 1, i) for i in (w.S_q - 1, w.S_q - 128, w.S_q - 129)]
    eo, el = sampled_rows_check(w, r, x.q, x.k, x.v, x.descale, tail)
    assert eo <= TOL_O[w.dtype] and el <= TOL_LSE, (eo, el)


@pytest.mark.parametrize("name", sorted(n for n, w in EXTRA_WORKLOADS.items() if not w.split and not w.bwd))
def test_gqa_workloads_sampled(name, cuda_lib):
    w = EXTRA_WORKLOADS[name]
    x = make_inputs(w, device="cuda")
    r = Run(w, x.q, x.k, x.v)
    torch.cuda.synchronize()
    assert r.status == 0 and r.device_status == 0 and r.guards_intact()
    assert _whole_output_finite(r)
    eo, el = sampled_rows_check(w, r, x.q, x.k, x.v, x.descale, _edge_rows(w, 96, seed=2))
    print(f"{name}: max|dO|={eo:.3g} max|dlse|={el:.3g}")
    assert eo <= TOL_O[w.dtype] and el <= TOL_LSE, (eo, el)
