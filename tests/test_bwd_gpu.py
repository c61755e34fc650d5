"""Backward pass (fa_bwd) against the float64 backward oracle.

Every element of dQ, dK and dV is held to the bound derived from the
kernels' arithmetic (tests/bwd_helpers.py), on shapes that span several tiles
with ragged tails in S_q and S_kv, causal and not, both layouts, fp16 and
bf16, D = 64 and 128, grouped-query heads, S_q != S_kv (including key tiles
no query sees), more work units than SMs (each CTA hands one unit's tiles
and accumulators over to the next), NaN-poisoned memory past the valid
rows, and a NaN-filled
workspace.  O and lse come from the oracle (rounded to the types a training
step passes) or, end to end, from the GPU forward pass.  Plus: canaries after
every output intact, no NaN / Inf, bit-identical repeat runs, argument
checks that launch nothing.
"""
import math

import numpy as np
import pytest
import torch

from oracle import backward as ob
from tiled_attention_10_gb300 import binding
from tiled_attention_10_gb300.inputs import BWD_WORKLOADS, Workload, make_dout, make_inputs
from tests.bwd_helpers import (SAFETY, U, BwdRun, bounds, head_bounds, make_do, oracle_o_lse,
                               to_bnsd64)
from tests.gpu_helpers import Run, to_device

pytestmark = pytest.mark.gpu


def _device_do(w, do_cpu):
    """dO on the device, keeping a NaN-poisoned tail after it when asked."""
    if not w.poison:
        return do_cpu.to("cuda")
    pad = 128 * w.H * w.D
    buf = torch.full((do_cpu.numel() + pad,), float("nan"), dtype=do_cpu.dtype, device="cuda")
    buf[: do_cpu.numel()] = do_cpu.reshape(-1).to("cuda")
    return buf[: do_cpu.numel()].view(do_cpu.shape)


def _check(w, r, ref, bnd):
    assert r.status == 0, binding.FA_STATUS.get(r.status)
    assert r.device_status == 0, binding.FA_STATUS.get(r.device_status)
    assert r.guards_intact(), "write past the end of dQ, dK or dV"
    worst = {}
    for name, got, want, b in zip(("dQ", "dK", "dV"), (r.dq, r.dk, r.dv), ref, bnd):
        g = to_bnsd64(got, w.layout)
        assert np.isfinite(g).all(), f"NaN/Inf in {name}"
        err = np.abs(g - want)
        ratio = err / b
        nrm = np.linalg.norm(want)
        rel = float(np.linalg.norm(g - want) / nrm) if nrm > 1e-6 else float("nan")
        worst[name] = (float(err.max()), float(ratio.max()), rel)
        bad = np.argwhere(ratio > 1.0)
        assert bad.size == 0, (f"{name}: {bad.shape[0]} elements over the bound, first {bad[0]}, "
                               f"err {err[tuple(bad[0])]:.3g} bound {b[tuple(bad[0])]:.3g}")
    return worst


def _run_case(w, end_to_end=False):
    x = make_inputs(w)
    do = make_do(w)
    ref_q, ref_k, ref_v, terms = ob.attention_bwd(
        x.q, x.k, x.v, do, dtype=w.dtype, layout=w.layout, B=w.B, H=w.H, S_q=w.S_q,
        S_kv=w.S_kv, D=w.D, scale=w.softmax_scale, causal=w.causal, H_kv=w.kv_heads,
        keep_terms=True)
    q, k, v = to_device(x)
    dod = _device_do(w, do)
    if end_to_end:
        f = Run(w, q, k, v)
        torch.cuda.synchronize()
        assert f.status == 0 and f.device_status == 0
        o, lse = f.o, f.lse
    else:
        o_cpu, lse_cpu = oracle_o_lse(w, terms)
        o, lse = o_cpu.to("cuda"), lse_cpu.to("cuda")
    r = BwdRun(w, q, k, v, o, dod, lse)
    torch.cuda.synchronize()
    o_in = to_bnsd64(o, w.layout)
    lse_in = lse.double().cpu().numpy()
    bnd = bounds(w, x, do, o_in, lse_in, terms, (ref_q, ref_k, ref_v))
    worst = _check(w, r, (ref_q, ref_k, ref_v), bnd)
    print(f"{w.B}x{w.H}/{w.kv_heads}x{w.S_q}x{w.S_kv}x{w.D} {w.dtype} {w.layout} "
          f"causal={w.causal}: " +
          ", ".join(f"{n} max|err|={e:.3g} max err/bound={rb:.3f} rel-rms={rr:.3g}"
                    for n, (e, rb, rr) in worst.items()))
    return r


CASES = [
    # B, H, H_kv, S_q, S_kv, D, dtype, layout, causal, poison
    (1, 2, 2, 256, 256, 128, "bf16", "BNSD", False, False),
    (1, 2, 2, 300, 300, 128, "bf16", "BNSD", True, False),
    (2, 4, 2, 200, 333, 64, "f16", "BSND", True, True),
    (1, 3, 3, 129, 1000, 64, "bf16", "BNSD", False, False),
    (1, 2, 1, 513, 257, 128, "f16", "BNSD", True, False),
    (1, 2, 2, 100, 400, 128, "bf16", "BSND", True, True),
    (2, 2, 2, 1, 1, 64, "bf16", "BNSD", False, False),
    (1, 1, 1, 1, 300, 128, "f16", "BNSD", True, False),
    (1, 8, 2, 640, 640, 128, "bf16", "BNSD", True, False),
    (1, 2, 2, 777, 129, 64, "bf16", "BSND", False, True),
    # more work units than SMs, so each CTA runs several in turn: 384 dQ
    # units and 96 dK/dV units of 4 query heads each ...
    (1, 32, 8, 1536, 1536, 64, "f16", "BSND", True, False),
    # ... and 400 dK/dV units of which 398 no query sees (zeros), taken
    # right after a unit with products by two of the CTAs
    (1, 2, 2, 128, 25600, 64, "bf16", "BNSD", True, False),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_bwd_parity(case, cuda_lib):
    B, H, H_kv, S_q, S_kv, D, dtype, layout, causal, poison = CASES[case]
    w = Workload("bwd", B, H, S_q, S_kv, D, dtype, layout, causal, seed=case + 1, H_kv=H_kv,
                 poison=poison)
    _run_case(w)


@pytest.mark.parametrize("dtype,causal", [("bf16", True), ("f16", False)])
def test_bwd_end_to_end_from_gpu_forward(dtype, causal, cuda_lib):
    w = Workload("bwd", 2, 4, 384, 384, 128, dtype, "BNSD", causal, seed=40)
    _run_case(w, end_to_end=True)


@pytest.mark.parametrize("dtype,causal,D", [("bf16", True, 128), ("f16", False, 64)])
def test_bwd_negative_scale(dtype, causal, D, cuda_lib):
    """A negative scale: S is computed as -Q K^T (and -K Q^T) with |scale| in
    the exponent, dQ and dK are multiplied by the signed scale."""
    w = Workload("bwd", 1, 4, 300, 300, D, dtype, "BNSD", causal, seed=21, H_kv=2,
                 scale=-1.0 / math.sqrt(D))
    _run_case(w)


def test_bwd_deterministic(cuda_lib):
    w = Workload("bwd", 1, 4, 520, 520, 128, "bf16", "BNSD", True, seed=7, H_kv=2)
    x = make_inputs(w)
    do = make_do(w).to("cuda")
    q, k, v = to_device(x)
    f = Run(w, q, k, v)
    torch.cuda.synchronize()
    r1 = BwdRun(w, q, k, v, f.o, do, f.lse)
    r2 = BwdRun(w, q, k, v, f.o, do, f.lse)
    torch.cuda.synchronize()
    for a, b in ((r1.dq, r2.dq), (r1.dk, r2.dk), (r1.dv, r2.dv)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bwd_bad_arguments_launch_nothing(cuda_lib):
    w = Workload("bwd", 1, 2, 128, 128, 128, "bf16", "BNSD", False, seed=3)
    x = make_inputs(w)
    q, k, v = to_device(x)
    do = make_do(w).to("cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 2, 128, device="cuda")
    dq, dk, dv = torch.full_like(q, 7.0), torch.full_like(k, 7.0), torch.full_like(v, 7.0)
    st, nbytes = binding.fa_bwd_workspace_size(1, 2, 128)
    ws = torch.empty(nbytes // 4 + 64, device="cuda")
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), 1, 2, 2, 128, 128, 128, w.softmax_scale,
            "BNSD", 0, "bf16", ws.data_ptr(), nbytes]
    bad = [
        (6, None, 1), (19, None, 1), (20, 16, 1), (19, ws.data_ptr() + 16, 3),
        (18, "e4m3", 2), (14, 96, 2), (3, o.data_ptr() + 2, 3), (11, 3, 1),
    ]
    for idx, val, code in bad:
        a = list(args)
        a[idx] = val
        assert binding.fa_bwd(*a) == code, (idx, val)
    torch.cuda.synchronize()
    assert bool((dq == 7.0).all()) and bool((dk == 7.0).all()) and bool((dv == 7.0).all())


def _head(t, layout, b, h):
    """One head of a device tensor as float64 numpy [S, D] (torch's exact
    upcast of the 16-bit values)."""
    x = t[b, h] if layout == "BNSD" else t[b, :, h]
    return x.double().cpu().numpy()


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(BWD_WORKLOADS))
def test_bwd_workload_sampled_heads(name, cuda_lib):
    """The measured backward workloads at full size, in the benchmark's launch
    configuration (O and lse from the GPU forward): every element of two
    key/value heads (the first and the last) against the oracle and the
    bound; no NaN / Inf anywhere; canaries intact."""
    w = BWD_WORKLOADS[name]
    x = make_inputs(w, device="cuda")
    do = make_dout(w, device="cuda")
    f = Run(w, x.q, x.k, x.v)
    torch.cuda.synchronize()
    assert f.status == 0 and f.device_status == 0
    r = BwdRun(w, x.q, x.k, x.v, f.o, do, f.lse)
    torch.cuda.synchronize()
    assert r.status == 0 and r.device_status == 0 and r.guards_intact()
    for t in (r.dq, r.dk, r.dv):
        assert bool(torch.isfinite(t.float()).all())
    g = w.H // w.kv_heads
    for (b, hk) in ((0, 0), (w.B - 1, w.kv_heads - 1)):
        k64, v64 = _head(x.k, w.layout, b, hk), _head(x.v, w.layout, b, hk)
        sum_dk = np.zeros_like(k64)
        sum_dv = np.zeros_like(v64)
        bnd_dk = np.zeros_like(k64)
        bnd_dv = np.zeros_like(v64)
        for h in range(hk * g, (hk + 1) * g):
            q64, do64 = _head(x.q, w.layout, b, h), _head(do, w.layout, b, h)
            t = ob.head_terms(q64, k64, v64, do64, w.softmax_scale, w.causal)
            o_in = _head(f.o, w.layout, b, h)
            lse_in = f.lse[b, h].double().cpu().numpy()
            b_dq, b_dk, b_dv = head_bounds(t, q64, k64, v64, do64, o_in, lse_in,
                                           w.softmax_scale, w.dtype)
            u = U[w.dtype] + 2.0 ** -24
            got = _head(r.dq, w.layout, b, h)
            lim = SAFETY * (b_dq + u * np.abs(t["dQ"]) + 2.0 ** -25)
            err = np.abs(got - t["dQ"])
            assert (err <= lim).all(), ("dQ", b, h, float((err / lim).max()))
            sum_dk += t["dK"]
            sum_dv += t["dV"]
            bnd_dk += b_dk
            bnd_dv += b_dv
        for nm, got_t, want, bb in (("dK", r.dk, sum_dk, bnd_dk), ("dV", r.dv, sum_dv, bnd_dv)):
            got = _head(got_t, w.layout, b, hk)
            lim = SAFETY * (bb + (U[w.dtype] + 2.0 ** -24) * np.abs(want) + 2.0 ** -25)
            err = np.abs(got - want)
            assert (err <= lim).all(), (nm, b, hk, float((err / lim).max()))
            print(f"{name} (b={b}, hk={hk}) {nm}: max|err|={err.max():.3g} "
                  f"max err/bound={(err / lim).max():.3f}")
