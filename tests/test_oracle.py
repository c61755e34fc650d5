"""Pins for the float64 oracle (CPU only).

The oracle is checked against things other than itself:
  * library routines that compute the same definition independently
    (torch's scaled_dot_product_attention and logsumexp in float64, numpy's
    and torch's own float16 / bfloat16 / float8_e4m3fn conversions);
  * closed forms worked out by hand for tiny inputs;
  * invariants of the definition (rows of P sum to one, linearity in V,
    permutation invariance, causal row i == attention over the prefix [0..i]).
The definition is the reference attention of "ops-transformer FlashAttention
build and tuning", section 4.3, with the safe-softmax max subtraction of
section 6.2 (FP16 overflow trap).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tiled_attention_10_gb300.inputs import Workload, make_inputs, shape_of

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _bnsd64(x: torch.Tensor, layout: str, descale: float = 1.0) -> torch.Tensor:
    """Library-side dequantisation to float64 BNSD (torch's own conversions)."""
    y = x.to(torch.float64) * descale
    return y if layout == "BNSD" else y.permute(0, 2, 1, 3).contiguous()


def _sdpa_ref(q, k, v, scale, causal):
    return F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)


def _all_rows(B, H, S):
    return np.array([(b, h, i) for b in range(B) for h in range(H) for i in range(S)], np.int64)


# ---------------------------------------------------------------------------
# Decoders vs library conversions, every code point.
# ---------------------------------------------------------------------------
def test_decode_f16_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(codes, "f16")
    ref = codes.view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[m], ref[m])


def test_decode_bf16_all_codes():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ours = oracle.decode(codes.numpy(), "bf16")
    ref = codes.view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[m], ref[m])


def test_decode_e4m3_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ours = oracle.decode(codes.numpy(), "e4m3")
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[m], ref[m])
    assert np.nanmax(ours) == 448.0 and np.isnan(ours).sum() == 2


# ---------------------------------------------------------------------------
# Against torch's float64 scaled_dot_product_attention (a library routine).
# ---------------------------------------------------------------------------
CASES = [
    # B, H, S_q, S_kv, D, dtype, layout, causal, scale
    (1, 1, 1, 1, 1, "bf16", "BNSD", False, 0.7),
    (2, 3, 5, 7, 4, "bf16", "BNSD", False, 0.5),
    (2, 3, 7, 5, 4, "f16", "BSND", True, 0.3),
    (1, 2, 6, 6, 3, "f16", "BNSD", True, 1.1),
    (2, 2, 9, 13, 8, "bf16", "BSND", False, None),
    (1, 3, 13, 9, 16, "bf16", "BNSD", True, None),
    (2, 1, 33, 40, 64, "f16", "BSND", True, 0.125),
    (1, 2, 17, 17, 128, "bf16", "BNSD", True, None),
]


@pytest.mark.parametrize("B,H,S_q,S_kv,D,dtype,layout,causal,scale", CASES)
def test_oracle_matches_torch_sdpa(B, H, S_q, S_kv, D, dtype, layout, causal, scale):
    w = Workload("t", B, H, S_q, S_kv, D, dtype, layout, causal, scale=scale, seed=S_q + D)
    x = make_inputs(w)
    O, lse = oracle.attention_full(x.q, x.k, x.v, dtype=dtype, layout=layout, B=B, H=H,
                                   S_q=S_q, S_kv=S_kv, D=D, scale=w.softmax_scale,
                                   causal=causal)
    q, k, v = (_bnsd64(t, layout) for t in (x.q, x.k, x.v))
    ref = _sdpa_ref(q, k, v, w.softmax_scale, causal).numpy()
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)
    s = w.softmax_scale * (q @ k.transpose(-1, -2))
    if causal:
        s = s.masked_fill(torch.ones(S_q, S_kv, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_oracle_fp8_descale_matches_torch_sdpa():
    """E4M3 inputs with per-tensor descales: the oracle works on value*descale."""
    w = Workload("t", 2, 2, 11, 19, 32, "e4m3", "BNSD", True, seed=5)
    x = make_inputs(w)
    assert all(d != 1.0 for d in x.descale)
    O, lse = oracle.attention_full(x.q, x.k, x.v, dtype="e4m3", layout="BNSD", B=2, H=2,
                                   S_q=11, S_kv=19, D=32, scale=w.softmax_scale, causal=True,
                                   descale=x.descale)
    q, k, v = (_bnsd64(t, "BNSD", d) for t, d in zip((x.q, x.k, x.v), x.descale))
    ref = _sdpa_ref(q, k, v, w.softmax_scale, True).numpy()
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)
    s = w.softmax_scale * (q @ k.transpose(-1, -2))
    s = s.masked_fill(torch.ones(11, 19, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def test_rows_entry_matches_full_entry():
    w = Workload("t", 2, 3, 21, 15, 8, "bf16", "BSND", True, seed=9)
    x = make_inputs(w)
    kw = dict(dtype="bf16", layout="BSND", B=2, H=3, S_q=21, S_kv=15, D=8,
              scale=w.softmax_scale, causal=True)
    O, lse = oracle.attention_full(x.q, x.k, x.v, **kw)
    rows = np.array([(1, 2, 20), (0, 0, 0), (1, 0, 7)], np.int64)
    Or, lr = oracle.attention_rows(x.q, x.k, x.v, rows=rows, **kw)
    for r, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(Or[r], O[b, h, i])
        assert lr[r] == lse[b, h, i]


# ---------------------------------------------------------------------------
# Closed forms, worked by hand.
# ---------------------------------------------------------------------------
def _run(q, k, v, scale, causal, dtype="f16", want_p=False):
    """Tiny single-head BNSD problem from float lists (exactly representable)."""
    tq = torch.tensor(q, dtype=torch.float64).to(torch.float16 if dtype == "f16" else torch.bfloat16)
    tk = torch.tensor(k, dtype=torch.float64).to(tq.dtype)
    tv = torch.tensor(v, dtype=torch.float64).to(tq.dtype)
    S_q, D = tq.shape
    S_kv = tk.shape[0]
    return oracle.attention_rows(tq, tk, tv, dtype=dtype, layout="BNSD", B=1, H=1, S_q=S_q,
                                 S_kv=S_kv, D=D, scale=scale, causal=causal,
                                 rows=_all_rows(1, 1, S_q), want_p=want_p)


def test_closed_form_two_keys_ln3():
    # S = [0, ln 3] -> P = [1/4, 3/4]; O = 4/4 + 3*8/4 = 7; lse = ln 4.
    O, lse = _run([[1.0]], [[0.0], [1.0]], [[4.0], [8.0]], scale=math.log(3.0), causal=False)
    assert abs(O[0, 0] - 7.0) < 1e-14
    assert abs(lse[0] - math.log(4.0)) < 1e-14


def test_closed_form_causal_two_rows():
    # q = [1,0], [1,0]; k = [1,0], [2,0]; scale = ln 2 -> S = [[ln2, 2 ln2], [ln2, 2 ln2]].
    # Row 0 sees only key 0: O = v0, lse = ln 2.  Row 1: P = [2/6, 4/6], lse = ln 6.
    O, lse, P = _run([[1.0, 0.0], [1.0, 0.0]], [[1.0, 0.0], [2.0, 0.0]], [[3.0, -1.0], [6.0, 5.0]],
                     scale=math.log(2.0), causal=True, want_p=True)
    np.testing.assert_allclose(O[0], [3.0, -1.0], atol=0)
    assert abs(lse[0] - math.log(2.0)) < 1e-15
    np.testing.assert_allclose(P[0], [1.0, 0.0], atol=0)
    np.testing.assert_allclose(P[1], [1 / 3, 2 / 3], atol=1e-15)
    np.testing.assert_allclose(O[1], [3.0 / 3 + 2 * 6.0 / 3, -1.0 / 3 + 2 * 5.0 / 3], atol=1e-14)
    assert abs(lse[1] - math.log(6.0)) < 1e-14


def test_closed_form_huge_logits_stay_finite():
    # The FP16 overflow trap (section 6.2): logits far above ln(65504) ~ 11.09 must
    # not overflow, so the max is subtracted before exp.
    # Equal scores 1000, 1000 -> plain mean, lse = 1000 + ln 2.
    O, lse = _run([[1.0]], [[1000.0], [1000.0]], [[4.0], [8.0]], scale=1.0, causal=False)
    assert abs(O[0, 0] - 6.0) < 1e-12 and abs(lse[0] - (1000.0 + math.log(2.0))) < 1e-12
    # Scores 1000, 1001 -> P = [1, e] / (1 + e), lse = 1001 + ln(1 + 1/e).
    O, lse = _run([[1.0]], [[1000.0], [1001.0]], [[4.0], [8.0]], scale=1.0, causal=False)
    e = math.e
    assert abs(O[0, 0] - (4.0 + 8.0 * e) / (1.0 + e)) < 1e-12
    assert abs(lse[0] - (1001.0 + math.log1p(1.0 / e))) < 1e-12


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(1)
    kr = rng.standard_normal(8).tolist()
    v = rng.standard_normal((9, 8)).round(3).tolist()
    q = rng.standard_normal((4, 8)).tolist()
    O, _ = _run(q, [kr] * 9, v, scale=0.37, causal=False, dtype="bf16")
    vv = torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).double().numpy()
    for i in range(4):
        np.testing.assert_allclose(O[i], vv.mean(0), atol=1e-14)


def test_constant_values_give_that_constant():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((5, 4)).tolist()
    k = rng.standard_normal((7, 4)).tolist()
    for causal in (False, True):
        O, _ = _run(q, k, [[1.5, -2.25, 0.5, 3.0]] * 7, scale=0.9, causal=causal)
        np.testing.assert_allclose(O, np.tile([1.5, -2.25, 0.5, 3.0], (5, 1)), atol=1e-14)


def test_dominant_logit_selects_its_value_row():
    # One key aligned with q at scale 64 vs others at most ~0: weight of the rest < e^-60.
    q = [[1.0, 0.0, 0.0, 0.0]]
    k = [[0.0, 1.0, 0.0, 0.0], [1.0, 0.0, 0.0, 0.0], [0.0, 0.0, -1.0, 0.0], [-1.0, 0.0, 0.0, 0.0]]
    v = [[1.0, 2.0, 3.0, 4.0], [-5.0, 6.0, -7.0, 8.0], [9.0, 9.0, 9.0, 9.0], [0.5, 0.5, 0.5, 0.5]]
    O, lse = _run(q, k, v, scale=64.0, causal=False)
    # |O - v[1]| <= 3 e^-64 * 20, far below one ulp: exact in float64.
    np.testing.assert_allclose(O[0], v[1], atol=1e-15, rtol=0)
    assert abs(lse[0] - 64.0) < 1e-14


def test_causal_row0_is_v0_and_lse_is_s00():
    w = Workload("t", 1, 2, 9, 9, 16, "bf16", "BSND", True, scale=0.25, seed=3)
    x = make_inputs(w)
    rows = np.array([(0, 0, 0), (0, 1, 0)], np.int64)
    O, lse = oracle.attention_rows(x.q, x.k, x.v, dtype="bf16", layout="BSND", B=1, H=2,
                                   S_q=9, S_kv=9, D=16, scale=0.25, causal=True, rows=rows)
    for r, h in enumerate((0, 1)):
        v0 = x.v[0, 0, h].double().numpy()
        np.testing.assert_array_equal(O[r], v0)
        s00 = 0.25 * float((x.q[0, 0, h].double() * x.k[0, 0, h].double()).sum())
        assert abs(lse[r] - s00) < 1e-15


def test_p_rows_sum_to_one_and_masked_entries_are_zero():
    w = Workload("t", 2, 2, 12, 10, 8, "f16", "BNSD", True, seed=4)
    x = make_inputs(w)
    O, lse, P = oracle.attention_rows(x.q, x.k, x.v, dtype="f16", layout="BNSD", B=2, H=2,
                                      S_q=12, S_kv=10, D=8, scale=w.softmax_scale, causal=True,
                                      rows=_all_rows(2, 2, 12), want_p=True)
    np.testing.assert_allclose(P.sum(1), 1.0, atol=1e-14)
    i = _all_rows(2, 2, 12)[:, 2]
    j = np.arange(10)
    assert (P[j[None, :] > i[:, None]] == 0).all()
    assert (P[j[None, :] <= i[:, None]] > 0).all()


def test_scale_zero_is_uniform_average():
    w = Workload("t", 1, 1, 6, 6, 4, "bf16", "BNSD", False, scale=0.0, seed=6)
    x = make_inputs(w)
    v = x.v[0, 0].double().numpy()
    for causal in (False, True):
        O, lse = oracle.attention_rows(x.q, x.k, x.v, dtype="bf16", layout="BNSD", B=1, H=1,
                                       S_q=6, S_kv=6, D=4, scale=0.0, causal=causal,
                                       rows=_all_rows(1, 1, 6))
        for i in range(6):
            n = i + 1 if causal else 6
            np.testing.assert_allclose(O[i], v[:n].mean(0), atol=1e-15)
            assert abs(lse[i] - math.log(n)) < 1e-15


def test_single_key_gives_v0():
    w = Workload("t", 2, 2, 5, 1, 8, "f16", "BSND", False, seed=7)
    x = make_inputs(w)
    O, _ = oracle.attention_full(x.q, x.k, x.v, dtype="f16", layout="BSND", B=2, H=2, S_q=5,
                                 S_kv=1, D=8, scale=0.5, causal=False)
    for b in range(2):
        for h in range(2):
            np.testing.assert_array_equal(O[b, h], np.tile(x.v[b, 0, h].double().numpy(), (5, 1)))


def test_linearity_in_v():
    w = Workload("t", 1, 1, 7, 9, 4, "bf16", "BNSD", True, seed=8)
    x = make_inputs(w)
    rng = np.random.default_rng(8)
    v1 = torch.tensor(rng.integers(-8, 8, (1, 1, 9, 4)), dtype=torch.bfloat16)
    v2 = torch.tensor(rng.integers(-8, 8, (1, 1, 9, 4)), dtype=torch.bfloat16)
    v3 = (3 * v1.double() - 2 * v2.double()).to(torch.bfloat16)  # exact in bf16
    kw = dict(dtype="bf16", layout="BNSD", B=1, H=1, S_q=7, S_kv=9, D=4, scale=0.4, causal=True)
    O1, _ = oracle.attention_full(x.q, x.k, v1, **kw)
    O2, _ = oracle.attention_full(x.q, x.k, v2, **kw)
    O3, _ = oracle.attention_full(x.q, x.k, v3, **kw)
    np.testing.assert_allclose(O3, 3 * O1 - 2 * O2, atol=1e-12)


def test_key_value_permutation_invariance_noncausal():
    w = Workload("t", 1, 2, 5, 11, 8, "f16", "BNSD", False, seed=10)
    x = make_inputs(w)
    perm = torch.randperm(11, generator=torch.Generator().manual_seed(0))
    kw = dict(dtype="f16", layout="BNSD", B=1, H=2, S_q=5, S_kv=11, D=8, scale=0.3, causal=False)
    O1, l1 = oracle.attention_full(x.q, x.k, x.v, **kw)
    O2, l2 = oracle.attention_full(x.q, x.k[:, :, perm].contiguous(), x.v[:, :, perm].contiguous(), **kw)
    np.testing.assert_allclose(O2, O1, atol=1e-14)
    np.testing.assert_allclose(l2, l1, atol=1e-14)


def test_causal_row_equals_noncausal_prefix():
    w = Workload("t", 1, 1, 8, 8, 4, "bf16", "BNSD", True, seed=11)
    x = make_inputs(w)
    O, lse = oracle.attention_full(x.q, x.k, x.v, dtype="bf16", layout="BNSD", B=1, H=1, S_q=8,
                                   S_kv=8, D=4, scale=0.6, causal=True)
    for i in range(8):
        Op, lp = oracle.attention_rows(x.q, x.k[:, :, : i + 1].contiguous(),
                                       x.v[:, :, : i + 1].contiguous(), dtype="bf16",
                                       layout="BNSD", B=1, H=1, S_q=8, S_kv=i + 1, D=4,
                                       scale=0.6, causal=False, rows=[(0, 0, i)])
        np.testing.assert_allclose(O[0, 0, i], Op[0], atol=1e-15)
        assert abs(lse[0, 0, i] - lp[0]) < 1e-15


def test_layouts_agree():
    w = Workload("t", 2, 3, 10, 12, 8, "bf16", "BNSD", True, seed=12)
    x = make_inputs(w)
    kw = dict(dtype="bf16", B=2, H=3, S_q=10, S_kv=12, D=8, scale=0.5, causal=True)
    O1, l1 = oracle.attention_full(x.q, x.k, x.v, layout="BNSD", **kw)
    t = [y.permute(0, 2, 1, 3).contiguous() for y in (x.q, x.k, x.v)]
    O2, l2 = oracle.attention_full(*t, layout="BSND", **kw)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(l1, l2)


def test_poisoned_tail_is_not_read():
    w = Workload("t", 2, 2, 9, 9, 8, "bf16", "BSND", True, poison=True, seed=13)
    x = make_inputs(w, pad_rows=4)
    assert torch.isnan(x.buffers[0][x.q.numel():].float()).all()
    O, lse = oracle.attention_full(x.q, x.k, x.v, dtype="bf16", layout="BSND", B=2, H=2, S_q=9,
                                   S_kv=9, D=8, scale=0.5, causal=True)
    assert np.isfinite(O).all() and np.isfinite(lse).all()


def test_argument_errors():
    z = np.zeros(16, np.uint16)
    with pytest.raises(ValueError):
        oracle.attention_rows(z, z, z, dtype="bf16", layout="BNSD", B=1, H=1, S_q=1, S_kv=0,
                              D=4, scale=1.0, causal=False, rows=[(0, 0, 0)])
    with pytest.raises(ValueError):
        oracle.attention_rows(z, z, z, dtype="bf16", layout="BNSD", B=1, H=1, S_q=2, S_kv=2,
                              D=4, scale=1.0, causal=False, rows=[(0, 0, 2)])


# ---------------------------------------------------------------------------
# Grouped-query attention: query head h reads key/value head h // (H // H_kv)
# (Q viewed as [.., H_kv, ngroups, D], the Hygon retrospective, defect 12).
# ---------------------------------------------------------------------------
GQA_CASES = [
    # B, H, H_kv, S_q, S_kv, D, dtype, layout, causal
    (1, 4, 2, 7, 9, 8, "bf16", "BNSD", False),
    (2, 6, 3, 11, 11, 16, "f16", "BSND", True),
    (1, 8, 1, 5, 13, 4, "bf16", "BSND", False),
    (2, 4, 4, 9, 6, 8, "bf16", "BNSD", True),
]


@pytest.mark.parametrize("B,H,H_kv,S_q,S_kv,D,dtype,layout,causal", GQA_CASES)
def test_gqa_matches_torch_sdpa_enable_gqa(B, H, H_kv, S_q, S_kv, D, dtype, layout, causal):
    w = Workload("t", B, H, S_q, S_kv, D, dtype, layout, causal, seed=H * 10 + H_kv, H_kv=H_kv)
    x = make_inputs(w)
    O, lse = oracle.attention_full(x.q, x.k, x.v, dtype=dtype, layout=layout, B=B, H=H,
                                   H_kv=H_kv, S_q=S_q, S_kv=S_kv, D=D, scale=w.softmax_scale,
                                   causal=causal)
    q, k, v = (_bnsd64(t, layout) for t in (x.q, x.k, x.v))
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=w.softmax_scale,
                                         enable_gqa=True).numpy()
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)
    kr = k.repeat_interleave(H // H_kv, dim=1)
    s = w.softmax_scale * (q @ kr.transpose(-1, -2))
    if causal:
        s = s.masked_fill(torch.ones(S_q, S_kv, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def test_gqa_head_mapping_is_floor_division():
    # K/V heads with constant, distinct values: query head h must see value h // 3.
    B, H, H_kv, S, D = 1, 6, 2, 4, 4
    q = torch.zeros(B, H, S, D, dtype=torch.bfloat16)
    k = torch.zeros(B, H_kv, S, D, dtype=torch.bfloat16)
    v = torch.stack([torch.full((S, D), float(c + 1)) for c in range(H_kv)]).unsqueeze(0)
    v = v.to(torch.bfloat16)
    O, _ = oracle.attention_full(q, k, v, dtype="bf16", layout="BNSD", B=B, H=H, H_kv=H_kv,
                                 S_q=S, S_kv=S, D=D, scale=1.0, causal=False)
    for h in range(H):
        assert (O[0, h] == float(h // 3 + 1)).all()


def test_gqa_rejects_non_multiple_heads():
    z = np.zeros(64, np.uint16)
    with pytest.raises(ValueError):
        oracle.attention_rows(z, z, z, dtype="bf16", layout="BNSD", B=1, H=3, H_kv=2, S_q=1,
                              S_kv=1, D=4, scale=1.0, causal=False, rows=[(0, 0, 0)])
