"""Shared helpers of the GPU tests: run the C-ABI call on seeded inputs and
compare with the float64 oracle.  (Test infrastructure; imports both sides.)"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tiled_attention_10_gb300 import binding
from tiled_attention_10_gb300.inputs import OUT_DTYPE, Workload, make_inputs, shape_of

# Max-abs tolerances on O per input type, and on lse.
TOL_O = {"f16": 4e-3, "bf16": 1.6e-2, "e4m3": 6e-2}
TOL_LSE = 1e-3
GUARD = 4096            # canary elements after O and lse
CANARY16 = 0x7BAD       # an unusual finite 16-bit pattern
CANARY32 = 0x7F7BAD00   # a finite fp32 pattern


def to_device(x, device="cuda"):
    """Copy inputs to the GPU keeping any NaN-poisoned tail right after the data."""
    out = []
    for t, buf in zip((x.q, x.k, x.v), x.buffers):
        if buf is t:
            out.append(t.to(device))
        else:
            b = buf.to(device)
            out.append(b[: t.numel()].view(t.shape))
    return out


class Run:
    """One fa_fwd call with guarded outputs."""

    def __init__(self, w: Workload, q, k, v, descale=None, stream=None):
        self.w = w
        dev = q.device
        oshape = shape_of(w.layout, w.B, w.H, w.S_q, w.D)
        n_o = int(np.prod(oshape))
        self.o_buf = torch.full((n_o + GUARD,), CANARY16, dtype=torch.int16, device=dev)
        self.o = self.o_buf[:n_o].view(OUT_DTYPE[w.dtype]).view(oshape)
        n_l = w.B * w.H * w.S_q
        self.l_buf = torch.full((n_l + GUARD,), CANARY32, dtype=torch.int32, device=dev)
        self.lse = self.l_buf[:n_l].view(torch.float32).view(w.B, w.H, w.S_q)
        ds = [None, None, None]
        self._ds = None
        if w.dtype == "e4m3" and descale is not None:
            self._ds = [torch.tensor([d], dtype=torch.float32, device=dev) for d in descale]
            ds = [t.data_ptr() for t in self._ds]
        if w.kv_heads == w.H:
            self.status = binding.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                         self.o.data_ptr(), self.lse.data_ptr(), w.B, w.H, w.S_q,
                                         w.S_kv, w.D, w.softmax_scale, w.layout, w.causal, w.dtype,
                                         ds[0], ds[1], ds[2], stream)
        else:
            self.status = binding.fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             self.o.data_ptr(), self.lse.data_ptr(), w.B, w.H,
                                             w.kv_heads, w.S_q, w.S_kv, w.D, w.softmax_scale,
                                             w.layout, w.causal, w.dtype, ds[0], ds[1], ds[2],
                                             stream)
        self.device_status = binding.fa_last_device_error(stream)

    def guards_intact(self) -> bool:
        n_o = self.o.numel()
        n_l = self.lse.numel()
        return bool((self.o_buf[n_o:] == CANARY16).all()) and bool((self.l_buf[n_l:] == CANARY32).all())

    def o_bnsd64(self) -> np.ndarray:
        o = self.o.float().cpu().double()
        if self.w.layout == "BSND":
            o = o.permute(0, 2, 1, 3)
        return o.contiguous().numpy()


def compare_full(w: Workload, r: Run, x):
    """Every row against the oracle; returns (max err O, max err lse)."""
    O, lse = oracle.attention_full(x.q, x.k, x.v, dtype=w.dtype, layout=w.layout, B=w.B, H=w.H,
                                   S_q=w.S_q, S_kv=w.S_kv, D=w.D, scale=w.softmax_scale,
                                   causal=w.causal, descale=x.descale, H_kv=w.kv_heads)
    og = r.o_bnsd64()
    lg = r.lse.cpu().double().numpy()
    return float(np.abs(og - O).max()), float(np.abs(lg - lse).max()), og, lg


def error_stats(got: np.ndarray, ref: np.ndarray, tol: float) -> dict:
    """The accuracy figures the Ascend page's verifier prints (section 4.3 of
    "ops-transformer FlashAttention build and tuning"): max and mean absolute
    difference, and how many elements lie within the tolerance."""
    d = np.abs(got - ref)
    return {"max_abs": float(d.max()), "mean_abs": float(d.mean()),
            "within_tol": int((d <= tol).sum()), "elements": int(d.size), "tol": tol}


def stats_line(name: str, so: dict, sl: dict) -> str:
    return (f"{name}: O max abs {so['max_abs']:.3g}, mean abs {so['mean_abs']:.3g}, "
            f"{so['within_tol']}/{so['elements']} within {so['tol']:g}; "
            f"lse max abs {sl['max_abs']:.3g}, mean abs {sl['mean_abs']:.3g}, "
            f"{sl['within_tol']}/{sl['elements']} within {sl['tol']:g}")


def check(w: Workload, r: Run, err_o: float, err_l: float, og=None, lg=None):
    assert r.status == 0, binding.FA_STATUS.get(r.status)
    assert r.device_status == 0, binding.FA_STATUS.get(r.device_status)
    assert r.guards_intact(), "write past the end of O or lse"
    if og is not None:
        assert np.isfinite(og).all() and np.isfinite(lg).all(), "NaN/Inf in outputs"
    assert err_o <= TOL_O[w.dtype], f"max |O - oracle| = {err_o:.3g} > {TOL_O[w.dtype]}"
    assert err_l <= TOL_LSE, f"max |lse - oracle| = {err_l:.3g} > {TOL_LSE}"


def run_small(w: Workload, pad_rows=128):
    x = make_inputs(w, pad_rows=pad_rows)
    q, k, v = to_device(x)
    r = Run(w, q, k, v, descale=x.descale)
    torch.cuda.synchronize()
    eo, el, og, lg = compare_full(w, r, x)
    check(w, r, eo, el, og, lg)
    return eo, el


def sampled_rows_check(w: Workload, r: Run, q, k, v, descale, rows):
    """Oracle on selected (b, h, i) rows using host copies of that head only."""
    err_o = err_l = 0.0
    og_all = []
    g = w.H // w.kv_heads
    for (b, h, i) in rows:
        hk = h // g   # key/value head of query head h
        if w.layout == "BNSD":
            qh, kh, vh = q[b, h].cpu(), k[b, hk].cpu(), v[b, hk].cpu()
            o_row = r.o[b, h, i].float().cpu().double().numpy()
        else:
            qh, kh, vh = q[b, :, h].cpu(), k[b, :, hk].cpu(), v[b, :, hk].cpu()
            o_row = r.o[b, i, h].float().cpu().double().numpy()
        O, lse = oracle.attention_rows(qh, kh, vh, dtype=w.dtype, layout="BNSD", B=1, H=1,
                                       S_q=w.S_q, S_kv=w.S_kv, D=w.D, scale=w.softmax_scale,
                                       causal=w.causal, rows=[(0, 0, int(i))], descale=descale)
        lg = float(r.lse[b, h, i].cpu())
        err_o = max(err_o, float(np.abs(o_row - O[0]).max()))
        err_l = max(err_l, abs(lg - float(lse[0])))
        og_all.append(o_row)
    return err_o, err_l
