"""float64 CPU oracle for the attention backward pass (gradients of the forward).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module; the product path never
imports it and shares no code with it.

What it computes.  The forward is the reference attention of the Ascend page
("ops-transformer FlashAttention build and tuning", section 4.3): for each
(batch, head), S = scale * Q K^T with the entries above the diagonal set to
-inf when causal (top-left aligned: query i sees key j iff j <= i), P = the
row softmax of S, O = P V.  The pages train with this operator (the mixed-
precision training configuration of the same page, and the backward dQ kernel
of the Hygon retrospective, defect 13) but print no backward formulas, so the
oracle is the chain rule through those three steps, written out:

    dV = P^T dO                       (O = P V)
    dP = dO V^T
    dS = P * (dP - rowsum(P * dP))    (Jacobian of the row softmax)
    dQ = scale * dS K,   dK = scale * dS^T Q

Masked entries have P = 0 and so get dS = 0.  Grouped-query attention
(H_kv < H): query head h reads key/value head h // (H // H_kv), so the
gradient of a key/value head is the sum over the query heads that read it.

Each step is one numpy float64 array operation on the materialised
S_q x S_kv matrices of one head -- no blocking, no fusion, no reordering.
The inputs are decoded exactly (f16 / bf16 values are exact in float64) with
the oracle's own decoder.
"""
from __future__ import annotations

import numpy as np

from . import decode


def _heads_bnsd(x, dtype, layout, B, heads, S, D) -> np.ndarray:
    """Decode a raw [B, heads, S, D] (BNSD) or [B, S, heads, D] (BSND) buffer
    to float64 in BNSD order."""
    a = decode(x, dtype).reshape(-1)[: B * heads * S * D]
    if layout == "BNSD":
        return a.reshape(B, heads, S, D)
    return a.reshape(B, S, heads, D).transpose(0, 2, 1, 3)


def _mask(S_q, S_kv, causal) -> np.ndarray:
    """True where query i may see key j."""
    if not causal:
        return np.ones((S_q, S_kv), dtype=bool)
    i = np.arange(S_q)[:, None]
    j = np.arange(S_kv)[None, :]
    return j <= i


def head_terms(q, k, v, do, scale, causal):
    """Forward and backward of one head, float64, every intermediate kept.

    q [S_q, D], k / v [S_kv, D], do [S_q, D].  Returns a dict with S, P, O,
    lse, dP, Dsum (= rowsum(P * dP)), dS, dQ, dK, dV.
    """
    S_q, S_kv = q.shape[0], k.shape[0]
    allowed = _mask(S_q, S_kv, causal)
    S = scale * (q @ k.T)
    S = np.where(allowed, S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=1, keepdims=True)
    P = E / l
    O = P @ v
    lse = (m + np.log(l))[:, 0]
    dV = P.T @ do
    dP = do @ v.T
    Dsum = (P * dP).sum(axis=1)
    dS = P * (dP - Dsum[:, None])
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    return dict(S=S, P=P, O=O, lse=lse, dP=dP, Dsum=Dsum, dS=dS, dQ=dQ, dK=dK, dV=dV)


def attention_bwd(q, k, v, do, *, dtype, layout, B, H, S_q, S_kv, D, scale, causal,
                  H_kv=None, kv_heads=None, keep_terms=False):
    """Gradients of the attention forward.

    q, do: raw buffers [B, H, S_q, D] (BNSD) or [B, S_q, H, D] (BSND); k, v:
    H_kv heads (default H).  Returns dQ [B, H, S_q, D], dK and dV
    [B, H_kv, S_kv, D] in BNSD order (float64).  With kv_heads = [(b, hk), ...]
    only those key/value heads and the query heads that read them are
    computed (the other entries are NaN).  With keep_terms the per-query-head
    intermediates of head_terms come back too, as a dict {(b, h): terms}.
    """
    H_kv = H if H_kv is None else H_kv
    g = H // H_kv
    Q = _heads_bnsd(q, dtype, layout, B, H, S_q, D)
    K = _heads_bnsd(k, dtype, layout, B, H_kv, S_kv, D)
    V = _heads_bnsd(v, dtype, layout, B, H_kv, S_kv, D)
    dO = _heads_bnsd(do, dtype, layout, B, H, S_q, D)
    dQ = np.full((B, H, S_q, D), np.nan)
    dK = np.full((B, H_kv, S_kv, D), np.nan)
    dV = np.full((B, H_kv, S_kv, D), np.nan)
    terms = {}
    todo = kv_heads if kv_heads is not None else [(b, hk) for b in range(B) for hk in range(H_kv)]
    for (b, hk) in todo:
        dK[b, hk] = 0.0
        dV[b, hk] = 0.0
        for h in range(hk * g, (hk + 1) * g):
            t = head_terms(Q[b, h], K[b, hk], V[b, hk], dO[b, h], scale, causal)
            dQ[b, h] = t["dQ"]
            dK[b, hk] += t["dK"]
            dV[b, hk] += t["dV"]
            if keep_terms:
                terms[(b, h)] = t
    if keep_terms:
        return dQ, dK, dV, terms
    return dQ, dK, dV
