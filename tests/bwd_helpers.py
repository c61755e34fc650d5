"""Backward-pass test helpers: running fa_bwd through the C ABI, and the
elementwise error bound the parity tests hold it to.

The bound is derived from the arithmetic the kernels perform, with the
oracle's float64 intermediates standing in for the exact values:

  * scores S = Q K^T accumulate D products in fp32 on the tensor cores (taken
    as n * 2^-23 * sum|terms| for an n-term sum, allowing truncating adds);
  * P = ex2(S * scale * log2(e) - lse * log2(e)) in fp32 (ex2.approx, relative
    error <= 2^-21), with the lse actually passed in (its own error included);
  * P rounded to the 16-bit type (unit roundoff u: 2^-8 bf16, 2^-11 fp16, plus
    2^-25 absolute for fp16 underflow) for dV = P^T dO;
  * dP = dO V^T in fp32; rowsum(dO * O) from the O actually passed in, fp32;
  * dS = P (dP - rowsum) in fp32, rounded to 16-bit for dK and dQ;
  * dV, dK, dQ accumulate in fp32 over S_q (times the group size for GQA) or
    S_kv terms, dK and dQ are multiplied by the scale in fp32, and all three
    are rounded to the 16-bit output type.

First-order terms only; the tests multiply the bound by 1.25 for the
second-order remainder.  No page fixes a backward tolerance: this is the one
the arithmetic gives.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import backward as ob
from tiled_attention_10_gb300 import binding
from tiled_attention_10_gb300.inputs import OUT_DTYPE, Workload, make_dout, shape_of

U = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}
A16 = {"bf16": 0.0, "f16": 2.0 ** -25}
GAM = 2.0 ** -23
EX2 = 2.0 ** -21
LOG2E = 1.0 / math.log(2.0)
SAFETY = 1.25

GUARD = 4096
CANARY16 = 0x7BAD


def head_bounds(t, q, k, v, do, o_in, lse_in, scale, dtype):
    """Bounds on |dQ|, |dK|, |dV| errors for one query head (dK, dV are this
    head's contributions).  q, do, o_in [S_q, D]; k, v [S_kv, D]; lse_in [S_q]
    (float64 copies of what the kernels read)."""
    u, a16 = U[dtype], A16[dtype]
    S_q, D = q.shape
    S_kv = k.shape[0]
    P, dP, Dsum, dS = t["P"], t["dP"], t["Dsum"], t["dS"]
    aq, ak, av, ado = np.abs(q), np.abs(k), np.abs(v), np.abs(do)
    vis = P > 0
    # exponent error of P (log2 units) -> relative error eta
    A = aq @ ak.T
    sl2 = abs(scale) * LOG2E                          # error terms scale with |scale|
    s2 = np.where(vis, t["S"] * LOG2E, 0.0)           # S * log2(e), S already scaled
    lse2 = lse_in * LOG2E
    x = np.where(vis, s2 - lse2[:, None], 0.0)
    dlse2 = np.abs(lse_in - t["lse"]) * LOG2E + np.abs(lse2) * 2.0 ** -23
    dx = sl2 * D * GAM * A + (np.abs(x) + np.abs(s2)) * 2.0 ** -23 + dlse2[:, None]
    eta = math.log(2.0) * dx + EX2
    eps_p16 = P * (eta + u) + a16 * vis               # P rounded to 16-bit
    # dV
    b_dv = eps_p16.T @ ado + S_q * GAM * (P.T @ ado)
    # rowsum(dO * O_in) and dP errors
    dD = (ado * np.abs(o_in - t["O"])).sum(axis=1) + D * 2.0 ** -24 * (ado * np.abs(o_in)).sum(axis=1)
    ddp = D * GAM * (ado @ av.T)
    g = np.abs(dP - Dsum[:, None])
    e_ds32 = P * eta * g + P * (ddp + dD[:, None]) * (1 + eta) + 2 * 2.0 ** -24 * P * g
    eps_ds16 = e_ds32 * (1 + u) + u * np.abs(dS) + a16 * vis
    ads = np.abs(dS)
    b_dk = abs(scale) * (eps_ds16.T @ aq + S_q * GAM * (ads.T @ aq))
    b_dq = abs(scale) * (eps_ds16 @ ak + S_kv * GAM * (ads @ ak))
    return b_dq, b_dk, b_dv


def bounds(w: Workload, x, do, o_in, lse_in, terms, ref):
    """Elementwise bounds for the whole problem (BNSD order, float64): dQ
    [B,H,S_q,D], dK / dV [B,H_kv,S_kv,D].  `terms` and `ref` = (dQ, dK, dV)
    from ob.attention_bwd; o_in [B,H,S_q,D] and lse_in [B,H,S_q] float64
    copies of the O and lse passed to the kernels.  Includes the output
    rounding (u |ref|, 2^-24 for the scale multiply, 2^-25 fp16 underflow)
    and the safety factor."""
    g = w.H // w.kv_heads
    Q = ob._heads_bnsd(x.q, w.dtype, w.layout, w.B, w.H, w.S_q, w.D)
    K = ob._heads_bnsd(x.k, w.dtype, w.layout, w.B, w.kv_heads, w.S_kv, w.D)
    V = ob._heads_bnsd(x.v, w.dtype, w.layout, w.B, w.kv_heads, w.S_kv, w.D)
    dO = ob._heads_bnsd(do, w.dtype, w.layout, w.B, w.H, w.S_q, w.D)
    bq = np.full((w.B, w.H, w.S_q, w.D), np.nan)
    bk = np.full((w.B, w.kv_heads, w.S_kv, w.D), np.nan)
    bv = np.full((w.B, w.kv_heads, w.S_kv, w.D), np.nan)
    for (b, h), t in terms.items():
        hk = h // g
        b_dq, b_dk, b_dv = head_bounds(t, Q[b, h], K[b, hk], V[b, hk], dO[b, h], o_in[b, h],
                                       lse_in[b, h], w.softmax_scale, w.dtype)
        bq[b, h] = b_dq
        if np.isnan(bk[b, hk]).all():
            bk[b, hk] = 0.0
            bv[b, hk] = 0.0
        bk[b, hk] += b_dk
        bv[b, hk] += b_dv
    out = []
    for bnd, r in zip((bq, bk, bv), ref):
        out.append(SAFETY * (bnd + (U[w.dtype] + 2.0 ** -24) * np.abs(r) + 2.0 ** -25))
    return tuple(out)


def to_bnsd64(t: torch.Tensor, layout: str) -> np.ndarray:
    y = t.float().cpu().double()
    if layout == "BSND":
        y = y.permute(0, 2, 1, 3)
    return y.contiguous().numpy()


class BwdRun:
    """fa_bwd on device inputs; gradients in guarded buffers (canaries after
    each), a NaN-filled workspace (its contents on entry must not matter)."""

    def __init__(self, w: Workload, q, k, v, o, do, lse, stream=None):
        dev = q.device
        self.w = w
        qshape = shape_of(w.layout, w.B, w.H, w.S_q, w.D)
        kshape = shape_of(w.layout, w.B, w.kv_heads, w.S_kv, w.D)
        self.bufs = []
        self.dq = self._guarded(qshape, w, dev)
        self.dk = self._guarded(kshape, w, dev)
        self.dv = self._guarded(kshape, w, dev)
        st, nbytes = binding.fa_bwd_workspace_size(w.B, w.H, w.S_q)
        assert st == 0
        self.ws = torch.full((nbytes // 4 + 64,), float("nan"), device=dev)
        self.status = binding.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     do.data_ptr(), lse.data_ptr(), self.dq.data_ptr(),
                                     self.dk.data_ptr(), self.dv.data_ptr(), w.B, w.H, w.kv_heads,
                                     w.S_q, w.S_kv, w.D, w.softmax_scale, w.layout, w.causal,
                                     w.dtype, self.ws.data_ptr(), self.ws.numel() * 4, stream)
        self.device_status = binding.fa_last_device_error(stream)

    def _guarded(self, shape, w, dev):
        n = int(np.prod(shape))
        buf = torch.full((n + GUARD,), CANARY16, dtype=torch.int16, device=dev)
        self.bufs.append((buf, n))
        return buf[:n].view(OUT_DTYPE[w.dtype]).view(shape)

    def guards_intact(self) -> bool:
        return all(bool((buf[n:] == CANARY16).all()) for buf, n in self.bufs)


def make_do(w: Workload, device="cpu"):
    """Upstream gradient dO (seeded, in q's shape and dtype)."""
    return make_dout(w, device=device)


def oracle_o_lse(w: Workload, terms):
    """O (rounded to the storage type, layout of q) and lse (fp32) from the
    oracle's float64 forward: the inputs a training step would pass."""
    O = np.zeros((w.B, w.H, w.S_q, w.D))
    L = np.zeros((w.B, w.H, w.S_q))
    for (b, h), t in terms.items():
        O[b, h] = t["O"]
        L[b, h] = t["lse"]
    o = torch.from_numpy(O).to(OUT_DTYPE[w.dtype])
    if w.layout == "BSND":
        o = o.permute(0, 2, 1, 3).contiguous()
    return o, torch.from_numpy(L).to(torch.float32)
