"""float64 CPU oracle for variable-length ("varlen") and paged-KV attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module; the product path never
imports it and shares no code with it.

Packed sequences.  Sequence s owns query rows [cu_q[s], cu_q[s+1]) of the
packed q / o ([total_q, H, D]) and, without paging, key rows
[cu_k[s], cu_k[s+1]) of the packed k / v ([total_k, H_kv, D]).  With paging
(the PagedAttention scheme of the Hygon retrospective, defect 11: logically
consecutive tokens in fixed-size physical pages addressed through a block
table), the cache is [num_pages, page_size, H_kv, D] and key j of sequence s
is row j % page_size of page block_table[s][j // page_size], for
j < seqused_k[s].

Each sequence is then ordinary attention (the reference attention of
"ops-transformer FlashAttention build and tuning", section 4.3) over its own
rows, one head at a time, with query head h reading key/value head
h // (H // H_kv).  Causal masks:
  mode 1 (top-left):     query i sees key j iff j <= i;
  mode 2 (bottom-right): query i sees key j iff j <= i + (S_kv - S_q), i.e.
                         the queries are the last S_q positions of the key
                         sequence (prefill after a cached prefix; decode).
A row that sees no key (possible only in mode 2 with S_q > S_kv, or with an
empty sequence) has O = 0 and lse = -inf.
"""
from __future__ import annotations

import numpy as np

from . import decode


def attend(q, k, v, scale, causal_mode):
    """One head of one sequence: q [S_q, D], k / v [S_kv, D] float64 ->
    (O [S_q, D], lse [S_q])."""
    S_q, S_kv = q.shape[0], k.shape[0]
    O = np.zeros((S_q, v.shape[1]))
    lse = np.full(S_q, -np.inf)
    if S_kv == 0 or S_q == 0:
        return O, lse
    S = scale * (q @ k.T)
    i = np.arange(S_q)[:, None]
    j = np.arange(S_kv)[None, :]
    if causal_mode == 1:
        allowed = j <= i
    elif causal_mode == 2:
        allowed = j <= i + (S_kv - S_q)
    else:
        allowed = np.ones((S_q, S_kv), dtype=bool)
    S = np.where(allowed, S, -np.inf)
    live = allowed.any(axis=1)
    m = np.where(live, S.max(axis=1), 0.0)
    E = np.where(allowed, np.exp(S - m[:, None]), 0.0)
    l = E.sum(axis=1)
    O[live] = (E[live] / l[live, None]) @ v
    lse[live] = m[live] + np.log(l[live])
    return O, lse


def _rows(x, dtype, heads, D, r0, r1):
    """Rows [r0, r1) of a packed [rows, heads, D] buffer, decoded to float64."""
    n = heads * D
    flat = x.reshape(-1) if hasattr(x, "reshape") else x
    return decode(flat[r0 * n: r1 * n], dtype).reshape(r1 - r0, heads, D)


def attention_varlen(q, k, v, *, cu_q, cu_k, H, H_kv, D, scale, causal_mode, dtype,
                     descale=(1.0, 1.0, 1.0), seqs=None):
    """Packed varlen attention.  q [total_q, H, D], k / v [total_k, H_kv, D]
    raw buffers; cu_q, cu_k int arrays of n_seqs + 1 offsets.  Returns
    O [total_q, H, D] and lse [H, total_q] (float64); with `seqs` only those
    sequences are computed (other rows NaN)."""
    total_q = q.numel() // (H * D) if hasattr(q, "numel") else q.size // (H * D)
    O = np.full((total_q, H, D), np.nan)
    L = np.full((H, total_q), np.nan)
    g = H // H_kv
    for s in (range(len(cu_q) - 1) if seqs is None else seqs):
        q0, q1, k0, k1 = int(cu_q[s]), int(cu_q[s + 1]), int(cu_k[s]), int(cu_k[s + 1])
        Q = _rows(q, dtype, H, D, q0, q1) * descale[0]
        K = _rows(k, dtype, H_kv, D, k0, k1) * descale[1]
        V = _rows(v, dtype, H_kv, D, k0, k1) * descale[2]
        for h in range(H):
            o, l = attend(Q[:, h], K[:, h // g], V[:, h // g], scale, causal_mode)
            O[q0:q1, h] = o
            L[h, q0:q1] = l
    return O, L


def gather_pages(cache, dtype, block_table, s, n_keys, page_size, H_kv, D):
    """Keys 0..n_keys-1 of sequence s from a paged cache [num_pages,
    page_size, H_kv, D]: row j % page_size of page block_table[s][j // page_size]."""
    page_elems = page_size * H_kv * D
    flat = cache.reshape(-1) if hasattr(cache, "reshape") else cache
    pages = {}
    out = np.empty((n_keys, H_kv, D))
    for j in range(n_keys):
        pid = int(block_table[s][j // page_size])
        if pid not in pages:
            pages[pid] = decode(flat[pid * page_elems:(pid + 1) * page_elems],
                                dtype).reshape(page_size, H_kv, D)
        out[j] = pages[pid][j % page_size]
    return out


def attention_paged(q, k_cache, v_cache, *, cu_q, seqused_k, block_table, page_size, H, H_kv,
                    D, scale, causal_mode, dtype, descale=(1.0, 1.0, 1.0), seqs=None):
    """Packed queries against a paged K/V cache.  Returns O [total_q, H, D]
    and lse [H, total_q] (float64)."""
    total_q = q.numel() // (H * D) if hasattr(q, "numel") else q.size // (H * D)
    O = np.full((total_q, H, D), np.nan)
    L = np.full((H, total_q), np.nan)
    g = H // H_kv
    for s in (range(len(cu_q) - 1) if seqs is None else seqs):
        q0, q1, n = int(cu_q[s]), int(cu_q[s + 1]), int(seqused_k[s])
        Q = _rows(q, dtype, H, D, q0, q1) * descale[0]
        K = gather_pages(k_cache, dtype, block_table, s, n, page_size, H_kv, D) * descale[1]
        V = gather_pages(v_cache, dtype, block_table, s, n, page_size, H_kv, D) * descale[2]
        for h in range(H):
            o, l = attend(Q[:, h], K[:, h // g], V[:, h // g], scale, causal_mode)
            O[q0:q1, h] = o
            L[h, q0:q1] = l
    return O, L
