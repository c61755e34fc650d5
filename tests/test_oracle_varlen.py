"""Pins for the varlen / paged-KV oracle (CPU only).

oracle/varlen.py is checked against:
  * torch's float64 scaled_dot_product_attention with an explicit boolean
    mask for each causal alignment (a library routine);
  * the C forward oracle (pinned to torch in test_oracle.py) run on each
    sequence of a packed batch on its own;
  * invariants of the paging scheme: a cache whose pages are in order gives
    the contiguous result; permuting the physical pages (and the block table
    with them) changes nothing;
  * closed forms: bottom-right alignment equals top-left when S_q == S_kv and
    equals no mask for a single query row (decode); rows that see no key
    give O = 0 and lse = -inf; a row that sees exactly key 0 gives V[0].
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import varlen as ov

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64)).to(torch.bfloat16)


def _torch_ref(q, k, v, scale, mode):
    S_q, S_kv = q.shape[0], k.shape[0]
    i = torch.arange(S_q)[:, None]
    j = torch.arange(S_kv)[None, :]
    if mode == 1:
        mask = j <= i
    elif mode == 2:
        mask = j <= i + (S_kv - S_q)
    else:
        mask = torch.ones(S_q, S_kv, dtype=torch.bool)
    Q, K, V = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    O = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask[None, None], scale=scale)[0, 0]
    S = scale * (torch.from_numpy(q) @ torch.from_numpy(k).T)
    lse = torch.logsumexp(S.masked_fill(~mask, float("-inf")), dim=1)
    return O.numpy(), lse.numpy()


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("S_q,S_kv", [(1, 1), (1, 9), (7, 7), (5, 12), (12, 5)])
def test_attend_matches_torch_masked_sdpa(mode, S_q, S_kv):
    g = np.random.default_rng(S_q * 10 + S_kv)
    q, k, v = g.standard_normal((S_q, 6)), g.standard_normal((S_kv, 6)), g.standard_normal((S_kv, 6))
    O, lse = ov.attend(q, k, v, 0.4, mode)
    live = np.isfinite(lse)
    tO, tl = _torch_ref(q, k, v, 0.4, mode)
    np.testing.assert_allclose(O[live], tO[live], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse[live], tl[live], rtol=1e-12, atol=1e-13)
    assert np.all(O[~live] == 0.0) and np.all(np.isneginf(lse[~live]))
    assert np.all(np.isneginf(tl[~live]))


def _packed(seq_q, seq_k, H, H_kv, D, seed):
    g = np.random.default_rng(seed)
    cu_q = np.concatenate([[0], np.cumsum(seq_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(seq_k)]).astype(np.int32)
    q = _bf16(g.standard_normal((int(cu_q[-1]), H, D)))
    k = _bf16(g.standard_normal((int(cu_k[-1]), H_kv, D)))
    v = _bf16(g.standard_normal((int(cu_k[-1]), H_kv, D)))
    return q, k, v, cu_q, cu_k


def test_varlen_equals_c_oracle_per_sequence():
    seq_q, seq_k = [5, 1, 17, 9], [5, 1, 17, 9]
    H, H_kv, D = 4, 2, 8
    q, k, v, cu_q, cu_k = _packed(seq_q, seq_k, H, H_kv, D, 1)
    for mode in (0, 1):
        O, L = ov.attention_varlen(q, k, v, cu_q=cu_q, cu_k=cu_k, H=H, H_kv=H_kv, D=D, scale=0.3,
                                   causal_mode=mode, dtype="bf16")
        for s in range(len(seq_q)):
            a, b = int(cu_q[s]), int(cu_q[s + 1])
            ka, kb = int(cu_k[s]), int(cu_k[s + 1])
            Oc, Lc = oracle.attention_full(q[a:b][None], k[ka:kb][None], v[ka:kb][None],
                                           dtype="bf16", layout="BSND", B=1, H=H, S_q=b - a,
                                           S_kv=kb - ka, D=D, scale=0.3, causal=bool(mode),
                                           H_kv=H_kv)
            np.testing.assert_allclose(O[a:b], Oc[0].transpose(1, 0, 2), rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(L[:, a:b], Lc[0], rtol=1e-12, atol=1e-13)


def _to_pages(k, seq_k, cu_k, page_size, H_kv, D, perm_seed=None):
    """Scatter packed keys into a paged cache; returns (cache, block_table)."""
    n_pages = [-(-n // page_size) for n in seq_k]
    total_pages = sum(n_pages) + 3
    phys = np.arange(total_pages)
    if perm_seed is not None:
        phys = np.random.default_rng(perm_seed).permutation(total_pages)
    cache = torch.full((total_pages, page_size, H_kv, D), float("nan"), dtype=torch.bfloat16)
    table = np.full((len(seq_k), max(n_pages)), 10 ** 6, dtype=np.int32)   # unused entries: junk
    nxt = 0
    for s, n in enumerate(seq_k):
        for p in range(n_pages[s]):
            pid = int(phys[nxt])
            nxt += 1
            table[s, p] = pid
            rows = k[int(cu_k[s]) + p * page_size: int(cu_k[s]) + min(n, (p + 1) * page_size)]
            cache[pid, : rows.shape[0]] = rows
    return cache, table


@pytest.mark.parametrize("page_size", [16, 64, 128])
@pytest.mark.parametrize("perm", [None, 5])
def test_paged_equals_contiguous(page_size, perm):
    seq_q, seq_k = [3, 1, 20], [40, 7, 150]
    H, H_kv, D = 4, 1, 8
    q, k, v, cu_q, cu_k = _packed(seq_q, seq_k, H, H_kv, D, 2)
    kc, table = _to_pages(k, seq_k, cu_k, page_size, H_kv, D, perm)
    vc, table_v = _to_pages(v, seq_k, cu_k, page_size, H_kv, D, perm)
    assert np.array_equal(table, table_v)
    for mode in (0, 2):
        O1, L1 = ov.attention_varlen(q, k, v, cu_q=cu_q, cu_k=cu_k, H=H, H_kv=H_kv, D=D,
                                     scale=0.5, causal_mode=mode, dtype="bf16")
        O2, L2 = ov.attention_paged(q, kc, vc, cu_q=cu_q, seqused_k=np.array(seq_k), block_table=table,
                                    page_size=page_size, H=H, H_kv=H_kv, D=D, scale=0.5,
                                    causal_mode=mode, dtype="bf16")
        np.testing.assert_array_equal(O1, O2)
        np.testing.assert_array_equal(L1, L2)


def test_bottom_right_special_cases():
    g = np.random.default_rng(3)
    q, k, v = g.standard_normal((6, 4)), g.standard_normal((6, 4)), g.standard_normal((6, 4))
    a = ov.attend(q, k, v, 0.7, 1)
    b = ov.attend(q, k, v, 0.7, 2)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    kk, vv = g.standard_normal((9, 4)), g.standard_normal((9, 4))
    c = ov.attend(q[:1], kk, vv, 0.7, 2)          # decode: one query sees every key
    d = ov.attend(q[:1], kk, vv, 0.7, 0)
    np.testing.assert_array_equal(c[0], d[0])
    np.testing.assert_array_equal(c[1], d[1])


def test_rows_without_keys():
    # S_q = 5, S_kv = 2, bottom-right: rows 0-2 see nothing, row 3 sees key 0.
    g = np.random.default_rng(4)
    q, k, v = g.standard_normal((5, 3)), g.standard_normal((2, 3)), g.standard_normal((2, 3))
    O, lse = ov.attend(q, k, v, 0.9, 2)
    assert np.all(O[:3] == 0.0) and np.all(np.isneginf(lse[:3]))
    np.testing.assert_allclose(O[3], v[0], rtol=1e-15)
    np.testing.assert_allclose(lse[3], 0.9 * q[3] @ k[0], rtol=1e-14)
    O0, l0 = ov.attend(q, k[:0], v[:0], 0.9, 0)  # an empty key sequence
    assert np.all(O0 == 0.0) and np.all(np.isneginf(l0))
