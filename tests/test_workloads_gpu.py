"""The five measured workloads at full size, in the launch configuration the
benchmark times, against the float64 oracle.

  fp16_1x8x512x64                  every element
  bf16_bsnd_causal_2x16x4097x64    every element (NaN-poisoned memory past the tail)
  bf16_4x32x4096x128               every element (after a fast pre-check of
                                   corner, tile-edge and random rows)
  fp8_causal_1x32x8192x128         every element (same pre-check)
  bf16_causal_16x64x16384x128      64 seeded (b, h, row) samples; each tensor
                                   holds 2^31 elements (> 4 GB)
Plus, at every size, properties that need no oracle: no NaN/Inf anywhere in
O or lse, canaries after the outputs intact.  The whole-output comparisons
print the figures the Ascend page's verifier reports: max and mean absolute
error and the count of elements within the tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_10_gb300.inputs import EXTRA_WORKLOADS, WORKLOADS, make_inputs, sample_rows
from tests.gpu_helpers import (TOL_LSE, TOL_O, Run, check, error_stats,
                               sampled_rows_check, stats_line, to_device)

pytestmark = pytest.mark.gpu


def _whole_output_finite(r: Run) -> bool:
    return bool(torch.isfinite(r.o.float()).all()) and bool(torch.isfinite(r.lse).all())


def _compare_every_element(w, r, x):
    """The whole output against the oracle (all heads, all rows); returns the
    error statistics of O and lse after asserting the tolerances."""
    O, L = oracle.attention_full(x.q, x.k, x.v, dtype=w.dtype, layout=w.layout, B=w.B, H=w.H,
                                 S_q=w.S_q, S_kv=w.S_kv, D=w.D, scale=w.softmax_scale,
                                 causal=w.causal, descale=x.descale, H_kv=w.kv_heads)
    og = r.o_bnsd64()
    lg = r.lse.cpu().double().numpy()
    assert np.isfinite(og).all() and np.isfinite(lg).all(), "NaN/Inf in outputs"
    so, sl = error_stats(og, O, TOL_O[w.dtype]), error_stats(lg, L, TOL_LSE)
    print(stats_line(w.name, so, sl))
    check(w, r, so["max_abs"], sl["max_abs"])
    assert so["within_tol"] == so["elements"] and sl["within_tol"] == sl["elements"]
    return so, sl


@pytest.mark.parametrize("name", ["fp16_1x8x512x64", "bf16_bsnd_causal_2x16x4097x64"])
def test_workload_every_row(name, cuda_lib):
    w = WORKLOADS[name]
    x = make_inputs(w)
    q, k, v = to_device(x)
    r = Run(w, q, k, v, descale=x.descale)
    torch.cuda.synchronize()
    _compare_every_element(w, r, x)


def _edge_rows(w, n_random, seed=0):
    rows = [tuple(int(v) for v in t) for t in sample_rows(w, n_random, seed)]
    S = w.S_q
    for i in (1, 127, 128, 129, 255, 256, S // 2, S - 129, S - 128, S - 2, S - 1):
        if 0 <= i < S:
            rows.append((w.B - 1, 0, i))
            rows.append((0, w.H - 1, i))
    return sorted(set(rows))


@pytest.mark.parametrize("name", ["bf16_4x32x4096x128", "fp8_causal_1x32x8192x128"])
def test_workload_every_element(name, cuda_lib):
    # The headline and the fp8 causal workload, whole: a fast pre-check of
    # edge and random rows, then every element of O and lse (16 to 30 s of
    # float64 oracle on the host cores).
    w = WORKLOADS[name]
    x = make_inputs(w, device="cuda")
    r = Run(w, x.q, x.k, x.v, descale=x.descale)
    torch.cuda.synchronize()
    assert r.status == 0 and r.device_status == 0 and r.guards_intact()
    assert _whole_output_finite(r)
    eo, el = sampled_rows_check(w, r, x.q, x.k, x.v, x.descale, _edge_rows(w, 64, seed=1))
    assert eo <= TOL_O[w.dtype] and el <= TOL_LSE, (eo, el)
    _compare_every_element(w, r, x)


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
