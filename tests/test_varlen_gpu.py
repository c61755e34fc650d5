"""Variable-length (fa_fwd_varlen) and paged-KV (fa_fwd_paged) forward passes
against the float64 varlen oracle, every row.

Packed batches mix empty, 1-row, tile-edge (127 / 128 / 129) and multi-tile
sequences; K lengths differ from Q lengths; all three causal settings;
bf16, fp16 and fp8; D = 64 and 128; grouped-query heads.  The paged cases use
page sizes 16 to 256 with the physical pages shuffled, junk in the unused
block-table entries and large finite junk in the unused slots of the last
pages.  O and lse carry canaries after them; rows that belong to no
sequence must stay untouched.
"""
import numpy as np
import pytest
import torch

from oracle import varlen as ov
from tiled_attention_10_gb300 import binding
from tiled_attention_10_gb300.inputs import OUT_DTYPE, TORCH_DTYPE, E4M3_MAX
from tests.gpu_helpers import CANARY16, CANARY32, GUARD, TOL_LSE, TOL_O

pytestmark = pytest.mark.gpu


def _rand(shape, dtype, g):
    x = torch.from_numpy(g.standard_normal(shape).astype(np.float32))
    if dtype != "e4m3":
        return x.to(TORCH_DTYPE[dtype]), 1.0
    amax = float(x.abs().max())
    d = amax / E4M3_MAX
    return (x / d).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn), d


class Out:
    def __init__(self, total_q, H, D, dtype, unused_rows=0):
        n_o = (total_q + unused_rows) * H * D
        self.o_buf = torch.full((n_o + GUARD,), CANARY16, dtype=torch.int16, device="cuda")
        self.o = self.o_buf[:n_o].view(OUT_DTYPE[dtype]).view(total_q + unused_rows, H, D)
        n_l = H * (total_q + unused_rows)
        self.l_buf = torch.full((n_l + GUARD,), CANARY32, dtype=torch.int32, device="cuda")
        self.lse = self.l_buf[:n_l].view(torch.float32).view(H, total_q + unused_rows)
        self.n_o, self.n_l = n_o, n_l

    def guards_intact(self):
        return bool((self.o_buf[self.n_o:] == CANARY16).all()) and \
            bool((self.l_buf[self.n_l:] == CANARY32).all())


def _compare(O, L, out, cu_q, dtype):
    og = out.o.float().cpu().double().numpy()
    lg = out.lse.cpu().double().numpy()
    covered = np.zeros(og.shape[0], dtype=bool)
    for s in range(len(cu_q) - 1):
        covered[int(cu_q[s]):int(cu_q[s + 1])] = True
    rows = np.nonzero(covered)[0]
    eo = float(np.abs(og[rows] - O[rows]).max()) if rows.size else 0.0
    ref_l, got_l = L[:, rows], lg[:, rows]
    assert np.array_equal(np.isneginf(ref_l), np.isneginf(got_l)), "rows without keys"
    fin = np.isfinite(ref_l)
    el = float(np.abs(got_l[fin] - ref_l[fin]).max()) if fin.any() else 0.0
    assert np.isfinite(og[rows]).all()
    assert eo <= TOL_O[dtype] and el <= TOL_LSE, (eo, el)
    # rows of no sequence: untouched
    raw = out.o.view(torch.int16).cpu().numpy()
    assert (raw[~covered] == CANARY16).all()
    return eo, el


def _descale_ptrs(ds, dtype):
    if dtype != "e4m3":
        return [], [None, None, None]
    keep = [torch.tensor([d], dtype=torch.float32, device="cuda") for d in ds]
    return keep, [t.data_ptr() for t in keep]


VARLEN_CASES = [
    # seq_q, seq_k, H, H_kv, D, dtype, causal
    ([5, 0, 1, 127, 128, 129, 300], [5, 0, 1, 127, 128, 129, 300], 4, 2, 128, "bf16", 1),
    ([5, 3, 200, 1], [9, 100, 150, 333], 2, 2, 64, "f16", 0),
    ([40, 1, 257, 130], [100, 700, 257, 65], 4, 1, 128, "bf16", 2),
    ([64, 260], [64, 513], 2, 2, 128, "e4m3", 2),
    ([300, 17], [300, 17], 8, 8, 64, "bf16", 1),
    # a negative scale (optional eighth field: the scale's sign)
    ([300, 17, 900], [300, 700, 900], 4, 2, 128, "bf16", 1, -1.0),
    ([64, 260], [64, 513], 2, 2, 128, "e4m3", 2, -1.0),
]


@pytest.mark.parametrize("case", range(len(VARLEN_CASES)))
def test_varlen_parity(case, cuda_lib):
    seq_q, seq_k, H, H_kv, D, dtype, causal, *sign = VARLEN_CASES[case]
    g = np.random.default_rng(100 + case)
    cu_q = np.concatenate([[0], np.cumsum(seq_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(seq_k)]).astype(np.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    q, dq = _rand((tq, H, D), dtype, g)
    k, dk = _rand((tk, H_kv, D), dtype, g)
    v, dv = _rand((tk, H_kv, D), dtype, g)
    scale = (sign[0] if sign else 1.0) / np.sqrt(D)
    O, L = ov.attention_varlen(q, k, v, cu_q=cu_q, cu_k=cu_k, H=H, H_kv=H_kv, D=D, scale=scale,
                               causal_mode=causal, dtype=dtype, descale=(dq, dk, dv))
    out = Out(tq, H, D, dtype, unused_rows=7)   # 7 trailing rows belong to no sequence
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    qpad = torch.zeros((tq + 7) * H * D, dtype=qd.dtype, device="cuda")
    qpad[: qd.numel()] = qd.reshape(-1)
    keep, ds = _descale_ptrs((dq, dk, dv), dtype)
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    st = binding.fa_fwd_varlen(qpad.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.o.data_ptr(),
                               out.lse.data_ptr(), cq.data_ptr(), ck.data_ptr(), len(seq_q),
                               tq + 7, tk, max(seq_q), H, H_kv, D, scale, causal, dtype, *ds)
    torch.cuda.synchronize()
    assert st == 0, binding.FA_STATUS.get(st)
    assert binding.fa_last_device_error() == 0
    assert out.guards_intact()
    O_full = np.concatenate([O, np.zeros((7, H, D))])
    L_full = np.concatenate([L, np.zeros((H, 7))], axis=1)
    eo, el = _compare(O_full, L_full, out, cu_q, dtype)
    print(f"varlen case {case}: max|dO|={eo:.3g} max|dlse|={el:.3g}")


def _paged_cache(k, seq_k, cu_k, page_size, H_kv, D, g, junk):
    """Pages shuffled; the unused slots of each last page hold finite junk."""
    n_pages = [max(1, -(-n // page_size)) for n in seq_k]
    total = sum(n_pages) + 5
    phys = g.permutation(total)
    cache = torch.empty((total, page_size, H_kv, D), dtype=k.dtype)
    cache.view(torch.uint8 if k.element_size() == 1 else torch.int16).copy_(
        junk(cache.shape).view(torch.uint8 if k.element_size() == 1 else torch.int16))
    table = np.full((len(seq_k), max(n_pages) + 2), 1 << 30, dtype=np.int32)  # junk entries
    nxt = 0
    for s, n in enumerate(seq_k):
        for pg in range(n_pages[s]):
            pid = int(phys[nxt])
            nxt += 1
            table[s, pg] = pid
            lo = int(cu_k[s]) + pg * page_size
            hi = int(cu_k[s]) + min(n, (pg + 1) * page_size)
            if hi > lo:
                cache[pid, : hi - lo] = k[lo:hi]
    return cache, table


PAGED_CASES = [
    # seq_q, seq_k, page_size, H, H_kv, D, dtype, causal
    ([1, 1, 1, 1], [1000, 17, 128, 257], 16, 8, 2, 128, "bf16", 2),    # decode
    ([100, 37], [600, 37], 64, 4, 4, 128, "bf16", 2),                  # prefix prefill
    ([128, 5, 1], [300, 129, 64], 32, 2, 1, 64, "f16", 0),
    ([200], [700], 256, 4, 2, 128, "bf16", 1),
    ([50, 3], [333, 1], 128, 2, 2, 128, "e4m3", 2),
]


@pytest.mark.parametrize("case", range(len(PAGED_CASES)))
def test_paged_parity(case, cuda_lib):
    seq_q, seq_k, page_size, H, H_kv, D, dtype, causal = PAGED_CASES[case]
    g = np.random.default_rng(200 + case)
    cu_q = np.concatenate([[0], np.cumsum(seq_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(seq_k)]).astype(np.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    q, dq = _rand((tq, H, D), dtype, g)
    k, dk = _rand((tk, H_kv, D), dtype, g)
    v, dv = _rand((tk, H_kv, D), dtype, g)

    def junk(shape):  # large finite values, in the storage type
        x = torch.from_numpy((g.standard_normal(shape) * 100).astype(np.float32))
        if dtype == "e4m3":
            return (x / dk).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
        return x.to(TORCH_DTYPE[dtype])

    kc, table = _paged_cache(k, seq_k, cu_k, page_size, H_kv, D, np.random.default_rng(7), junk)
    vc, table_v = _paged_cache(v, seq_k, cu_k, page_size, H_kv, D, np.random.default_rng(7), junk)
    assert np.array_equal(table, table_v)
    scale = 1.0 / np.sqrt(D)
    O, L = ov.attention_paged(q, kc, vc, cu_q=cu_q, seqused_k=np.array(seq_k), block_table=table,
                              page_size=page_size, H=H, H_kv=H_kv, D=D, scale=scale,
                              causal_mode=causal, dtype=dtype, descale=(dq, dk, dv))
    out = Out(tq, H, D, dtype)
    keep, ds = _descale_ptrs((dq, dk, dv), dtype)
    cq = torch.from_numpy(cu_q).cuda()
    sk = torch.tensor(seq_k, dtype=torch.int32, device="cuda")
    tb = torch.from_numpy(table).cuda()
    qd, kcd, vcd = q.cuda(), kc.cuda(), vc.cuda()
    st = binding.fa_fwd_paged(qd.data_ptr(), kcd.data_ptr(), vcd.data_ptr(), out.o.data_ptr(),
                              out.lse.data_ptr(), cq.data_ptr(), sk.data_ptr(), tb.data_ptr(),
                              len(seq_q), table.shape[1], page_size, kc.shape[0], tq, max(seq_q),
                              H, H_kv, D, scale, causal, dtype, *ds)
    torch.cuda.synchronize()
    assert st == 0, binding.FA_STATUS.get(st)
    assert binding.fa_last_device_error() == 0
    assert out.guards_intact()
    eo, el = _compare(O, L, out, cu_q, dtype)
    print(f"paged case {case} (page {page_size}): max|dO|={eo:.3g} max|dlse|={el:.3g}")


def test_varlen_matches_dense_call(cuda_lib):
    # One sequence per batch entry with equal lengths: the packed call must
    # give the dense BSND call's bits.
    B, S, H, D = 3, 300, 4, 128
    g = np.random.default_rng(9)
    q, _ = _rand((B, S, H, D), "bf16", g)
    k, _ = _rand((B, S, H, D), "bf16", g)
    v, _ = _rand((B, S, H, D), "bf16", g)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1 = torch.empty_like(qd)
    l1 = torch.empty(B, H, S, device="cuda")
    assert binding.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o1.data_ptr(), l1.data_ptr(),
                          B, H, S, S, D, 0.1, "BSND", 1, "bf16", None, None, None) == 0
    o2 = torch.empty_like(qd)
    l2 = torch.empty(H, B * S, device="cuda")
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device="cuda")
    assert binding.fa_fwd_varlen(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o2.data_ptr(),
                                 l2.data_ptr(), cu.data_ptr(), cu.data_ptr(), B, B * S, B * S, S,
                                 H, H, D, 0.1, 1, "bf16") == 0
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.permute(1, 0, 2).reshape(H, B * S), l2)


def test_varlen_host_checks(cuda_lib):
    t = torch.zeros(1024, device="cuda")
    a = t.data_ptr()
    base = dict(q=a, k=a, v=a, o=a, lse=a, cu_q=a, cu_k=a, n_seqs=1, total_q=4, total_k=4,
                max_seqlen_q=4, H=2, H_kv=2, D=64, scale=0.1, causal=0, dtype="bf16")

    def call(**kw):
        x = {**base, **kw}
        return binding.fa_fwd_varlen(x["q"], x["k"], x["v"], x["o"], x["lse"], x["cu_q"], x["cu_k"],
                                     x["n_seqs"], x["total_q"], x["total_k"], x["max_seqlen_q"],
                                     x["H"], x["H_kv"], x["D"], x["scale"], x["causal"], x["dtype"])
    assert call(cu_q=None) == 1
    assert call(n_seqs=0) == 1
    assert call(causal=3) == 1
    assert call(max_seqlen_q=0) == 1
    assert call(D=96) == 2
    assert call(cu_k=a + 2) == 3
    assert call(total_q=0) == 0            # nothing to do
    assert binding.fa_fwd_paged(a, a, a, a, a, a, a, a, 1, 1, 48, 4, 4, 4, 2, 2, 64, 0.1, 0,
                                "bf16") == 2    # page size 48
    assert binding.fa_fwd_paged(a, a, a, a, a, a, a, None, 1, 1, 64, 4, 4, 4, 2, 2, 64, 0.1, 0,
                                "bf16") == 1    # no block table
    assert binding.fa_fwd_paged(a, a, a, a, a, a, a, a, 1, 0, 64, 4, 4, 4, 2, 2, 64, 0.1, 0,
                                "bf16") == 1    # max pages 0


def _paged_setup(case):
    seq_q, seq_k, page_size, H, H_kv, D, dtype, causal = PAGED_CASES[case]
    g = np.random.default_rng(200 + case)
    cu_q = np.concatenate([[0], np.cumsum(seq_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(seq_k)]).astype(np.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    q, dq = _rand((tq, H, D), dtype, g)
    k, dk = _rand((tk, H_kv, D), dtype, g)
    v, dv = _rand((tk, H_kv, D), dtype, g)

    def junk(shape):
        x = torch.from_numpy((g.standard_normal(shape) * 100).astype(np.float32))
        if dtype == "e4m3":
            return (x / dk).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
        return x.to(TORCH_DTYPE[dtype])

    kc, table = _paged_cache(k, seq_k, cu_k, page_size, H_kv, D, np.random.default_rng(7), junk)
    vc, _ = _paged_cache(v, seq_k, cu_k, page_size, H_kv, D, np.random.default_rng(7), junk)
    return dict(seq_q=seq_q, seq_k=seq_k, page_size=page_size, H=H, H_kv=H_kv, D=D, dtype=dtype,
                causal=causal, cu_q=cu_q, tq=tq, q=q, kc=kc, vc=vc, table=table,
                descale=(dq, dk, dv))


@pytest.mark.parametrize("n_splits", [1, 2, 3, 7])
@pytest.mark.parametrize("case", range(len(PAGED_CASES)))
def test_paged_split_parity(case, n_splits, cuda_lib):
    c = _paged_setup(case)
    scale = 1.0 / np.sqrt(c["D"])
    O, L = ov.attention_paged(c["q"], c["kc"], c["vc"], cu_q=c["cu_q"],
                              seqused_k=np.array(c["seq_k"]), block_table=c["table"],
                              page_size=c["page_size"], H=c["H"], H_kv=c["H_kv"], D=c["D"],
                              scale=scale, causal_mode=c["causal"], dtype=c["dtype"],
                              descale=c["descale"])
    out = Out(c["tq"], c["H"], c["D"], c["dtype"])
    keep, ds = _descale_ptrs(c["descale"], c["dtype"])
    st, nb = binding.fa_fwd_paged_split_workspace_size(c["H"], c["tq"], c["D"], n_splits,
                                                       len(c["seq_q"]))
    assert st == 0
    ws = torch.full((nb // 4 + 64,), float("nan"), device="cuda")   # contents must not matter
    cq = torch.from_numpy(c["cu_q"]).cuda()
    sk = torch.tensor(c["seq_k"], dtype=torch.int32, device="cuda")
    tb = torch.from_numpy(c["table"]).cuda()
    qd, kcd, vcd = c["q"].cuda(), c["kc"].cuda(), c["vc"].cuda()
    st = binding.fa_fwd_paged_split(qd.data_ptr(), kcd.data_ptr(), vcd.data_ptr(),
                                    out.o.data_ptr(), out.lse.data_ptr(), cq.data_ptr(),
                                    sk.data_ptr(), tb.data_ptr(), len(c["seq_q"]),
                                    c["table"].shape[1], c["page_size"], c["kc"].shape[0], c["tq"],
                                    max(c["seq_q"]), c["H"], c["H_kv"], c["D"], scale, c["causal"],
                                    c["dtype"], *ds, n_splits, ws.data_ptr(), ws.numel() * 4)
    torch.cuda.synchronize()
    assert st == 0, binding.FA_STATUS.get(st)
    assert binding.fa_last_device_error() == 0
    assert out.guards_intact()
    eo, el = _compare(O, L, out, c["cu_q"], c["dtype"])
    print(f"paged split case {case} n_splits={n_splits}: max|dO|={eo:.3g} max|dlse|={el:.3g}")


def test_paged_sequence_order(cuda_lib):
    # fa_fwd_paged_split with a workspace first ranks the sequences longest
    # first (int32 [n_seqs] at the workspace's start) and hands out work in
    # that order; the order moves work between CTAs but not its arithmetic, so
    # the outputs equal fa_fwd_paged's bits.  Ties keep the given order.
    c = _paged_setup(0)
    seq_k = [1000, 17, 128, 257]
    assert list(c["seq_k"]) == seq_k
    scale = 1.0 / np.sqrt(c["D"])
    cq = torch.from_numpy(c["cu_q"]).cuda()
    sk = torch.tensor(seq_k, dtype=torch.int32, device="cuda")
    tb = torch.from_numpy(c["table"]).cuda()
    qd, kcd, vcd = c["q"].cuda(), c["kc"].cuda(), c["vc"].cuda()
    keep, ds = _descale_ptrs(c["descale"], c["dtype"])
    args = (len(c["seq_q"]), c["table"].shape[1], c["page_size"], c["kc"].shape[0], c["tq"],
            max(c["seq_q"]), c["H"], c["H_kv"], c["D"], scale, c["causal"], c["dtype"], *ds)
    ref = Out(c["tq"], c["H"], c["D"], c["dtype"])
    assert binding.fa_fwd_paged(qd.data_ptr(), kcd.data_ptr(), vcd.data_ptr(), ref.o.data_ptr(),
                                ref.lse.data_ptr(), cq.data_ptr(), sk.data_ptr(), tb.data_ptr(),
                                *args) == 0
    st, nb = binding.fa_fwd_paged_split_workspace_size(c["H"], c["tq"], c["D"], 1, len(seq_k))
    assert st == 0 and nb == 256                       # the order alone, one aligned block
    ws = torch.full((nb // 4,), -7, dtype=torch.int32, device="cuda")
    out = Out(c["tq"], c["H"], c["D"], c["dtype"])
    assert binding.fa_fwd_paged_split(qd.data_ptr(), kcd.data_ptr(), vcd.data_ptr(),
                                      out.o.data_ptr(), out.lse.data_ptr(), cq.data_ptr(),
                                      sk.data_ptr(), tb.data_ptr(), *args, 1, ws.data_ptr(),
                                      nb) == 0
    torch.cuda.synchronize()
    assert binding.fa_last_device_error() == 0
    assert ws[:4].tolist() == [0, 3, 2, 1]             # 1000, 257, 128, 17 keys
    assert torch.equal(out.o.view(torch.int16), ref.o.view(torch.int16))
    assert torch.equal(out.lse, ref.lse)
    # equal lengths keep their index order; lengths past the cache are clamped
    sk2 = torch.tensor([128, 9999999, 128, 17], dtype=torch.int32, device="cuda")
    out2 = Out(c["tq"], c["H"], c["D"], c["dtype"])
    assert binding.fa_fwd_paged_split(qd.data_ptr(), kcd.data_ptr(), vcd.data_ptr(),
                                      out2.o.data_ptr(), out2.lse.data_ptr(), cq.data_ptr(),
                                      sk2.data_ptr(), tb.data_ptr(), *args, 1, ws.data_ptr(),
                                      nb) == 0
    torch.cuda.synchronize()
    assert binding.fa_last_device_error() == 0
    assert ws[:4].tolist() == [1, 0, 2, 3]


@pytest.mark.parametrize("n_seqs", [16384, 16385])
def test_paged_split_many_sequences(n_seqs, cuda_lib):
    # Decode over the largest batch that is still ordered (16384 sequences) and
    # one past it (given order, no order in the workspace: the partials start at
    # its beginning).  Sampled sequences against the oracle; the written order
    # against a host sort.
    H, H_kv, D, page_size, dtype = 8, 2, 64, 16, "bf16"
    g = np.random.default_rng(n_seqs)
    seq_q = [1] * n_seqs
    seq_k = [int(x) for x in g.integers(1, 41, n_seqs)]
    cu_q = np.arange(n_seqs + 1, dtype=np.int32)
    cu_k = np.concatenate([[0], np.cumsum(seq_k)]).astype(np.int32)
    q, _ = _rand((n_seqs, H, D), dtype, g)
    k, _ = _rand((int(cu_k[-1]), H_kv, D), dtype, g)
    v, _ = _rand((int(cu_k[-1]), H_kv, D), dtype, g)
    junk = lambda shape: torch.from_numpy(g.standard_normal(shape).astype(np.float32)).to(
        TORCH_DTYPE[dtype])
    kc, table = _paged_cache(k, seq_k, cu_k, page_size, H_kv, D, np.random.default_rng(1), junk)
    vc, _ = _paged_cache(v, seq_k, cu_k, page_size, H_kv, D, np.random.default_rng(1), junk)
    scale = 1.0 / np.sqrt(D)
    n_splits = 2
    st, nb = binding.fa_fwd_paged_split_workspace_size(H, n_seqs, D, n_splits, n_seqs)
    assert st == 0
    ws = torch.full((nb // 4 + 64,), float("nan"), device="cuda")
    out = Out(n_seqs, H, D, dtype)
    cq = torch.from_numpy(cu_q).cuda()
    sk = torch.tensor(seq_k, dtype=torch.int32, device="cuda")
    tb = torch.from_numpy(table).cuda()
    qd, kcd, vcd = q.cuda(), kc.cuda(), vc.cuda()   # held until the call has run
    st = binding.fa_fwd_paged_split(qd.data_ptr(), kcd.data_ptr(),
                                    vcd.data_ptr(), out.o.data_ptr(), out.lse.data_ptr(),
                                    cq.data_ptr(), sk.data_ptr(), tb.data_ptr(), n_seqs,
                                    table.shape[1], page_size, kc.shape[0], n_seqs, 1, H, H_kv, D,
                                    scale, 2, dtype, None, None, None, n_splits, ws.data_ptr(),
                                    ws.numel() * 4)
    torch.cuda.synchronize()
    assert st == 0, binding.FA_STATUS.get(st)
    assert binding.fa_last_device_error() == 0
    assert out.guards_intact()
    if n_seqs <= 16384:
        want = np.lexsort((np.arange(n_seqs), -np.array(seq_k)))   # longest first, then index
        assert np.array_equal(ws.view(torch.int32)[:n_seqs].cpu().numpy(), want)
    pick = np.sort(np.concatenate([[0, n_seqs - 1], g.choice(n_seqs, 30, replace=False)]))
    O, L = ov.attention_paged(q[torch.from_numpy(pick)], kc, vc, cu_q=np.arange(len(pick) + 1, dtype=np.int32),
                              seqused_k=np.array(seq_k)[pick], block_table=table[pick],
                              page_size=page_size, H=H, H_kv=H_kv, D=D, scale=scale,
                              causal_mode=2, dtype=dtype, descale=(1.0, 1.0, 1.0))
    og = out.o[torch.from_numpy(pick).cuda()].float().cpu().double().numpy()
    lg = out.lse[:, torch.from_numpy(pick).cuda()].cpu().double().numpy()
    assert np.abs(og - O).max() <= TOL_O[dtype] and np.abs(lg - L).max() <= TOL_LSE


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_paged_split_planned(dtype, cuda_lib):
    # Decode with the split count fa_fwd_paged_split_plan picks for this
    # device: a few sequences of very different lengths leave most SMs idle,
    # so it splits many ways (up to half the longest sequence's blocks).
    H, H_kv, D, page_size = 8, 2, 128, 64
    g = np.random.default_rng(5)
    seq_k = [5000, 37, 1200, 129, 3100, 640]
    n_seqs = len(seq_k)
    cu_q = np.arange(n_seqs + 1, dtype=np.int32)
    cu_k = np.concatenate([[0], np.cumsum(seq_k)]).astype(np.int32)
    q, dq = _rand((n_seqs, H, D), dtype, g)
    k, dk = _rand((int(cu_k[-1]), H_kv, D), dtype, g)
    v, dv = _rand((int(cu_k[-1]), H_kv, D), dtype, g)

    def junk(shape):
        x = torch.from_numpy((g.standard_normal(shape) * 100).astype(np.float32))
        if dtype == "e4m3":
            return (x / dk).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
        return x.to(TORCH_DTYPE[dtype])

    kc, table = _paged_cache(k, seq_k, cu_k, page_size, H_kv, D, np.random.default_rng(2), junk)
    vc, _ = _paged_cache(v, seq_k, cu_k, page_size, H_kv, D, np.random.default_rng(2), junk)
    st, n_splits, nb = binding.fa_fwd_paged_split_plan(n_seqs, n_seqs, 1, sum(seq_k), max(seq_k),
                                                       H, H_kv, D)
    assert st == 0 and 2 <= n_splits <= 32
    assert nb == binding.fa_fwd_paged_split_workspace_size(H, n_seqs, D, n_splits, n_seqs)[1]
    ws = torch.full((nb // 4 + 64,), float("nan"), device="cuda")
    out = Out(n_seqs, H, D, dtype)
    scale = 1.0 / np.sqrt(D)
    ds, dst = [None] * 3, []
    if dtype == "e4m3":
        dst = [torch.tensor([d], dtype=torch.float32, device="cuda") for d in (dq, dk, dv)]
        ds = [t.data_ptr() for t in dst]
    cq = torch.from_numpy(cu_q).cuda()
    sk = torch.tensor(seq_k, dtype=torch.int32, device="cuda")
    tb = torch.from_numpy(table).cuda()
    qd, kcd, vcd = q.cuda(), kc.cuda(), vc.cuda()   # held until the call has run
    st = binding.fa_fwd_paged_split(qd.data_ptr(), kcd.data_ptr(), vcd.data_ptr(),
                                    out.o.data_ptr(), out.lse.data_ptr(), cq.data_ptr(),
                                    sk.data_ptr(), tb.data_ptr(), n_seqs, table.shape[1],
                                    page_size, kc.shape[0], n_seqs, 1, H, H_kv, D, scale, 2,
                                    dtype, *ds, n_splits, ws.data_ptr(), ws.numel() * 4)
    torch.cuda.synchronize()
    assert st == 0, binding.FA_STATUS.get(st)
    assert binding.fa_last_device_error() == 0
    assert out.guards_intact()
    O, L = ov.attention_paged(q, kc, vc, cu_q=cu_q, seqused_k=np.array(seq_k), block_table=table,
                              page_size=page_size, H=H, H_kv=H_kv, D=D, scale=scale,
                              causal_mode=2, dtype=dtype, descale=(dq, dk, dv))
    eo = np.abs(out.o.float().cpu().double().numpy() - O).max()
    el = np.abs(out.lse.cpu().double().numpy() - L).max()
    print(f"planned paged split ({dtype}): n_splits={n_splits} max|dO|={eo:.3g} max|dlse|={el:.3g}")
    assert eo <= TOL_O[dtype] and el <= TOL_LSE
