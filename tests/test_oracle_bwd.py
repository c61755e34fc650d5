"""Pins for the float64 backward oracle (CPU only).

The backward oracle (oracle/backward.py) is the chain rule through the forward
reference attention.  It is checked against things other than itself:
  * torch autograd through torch's float64 scaled_dot_product_attention (a
    library routine computing the same gradients independently), with causal
    masks, both layouts, S_q != S_kv and grouped-query heads;
  * central finite differences of the forward (its forward is first pinned
    to the C forward oracle, which is pinned to torch in test_oracle.py);
  * closed forms and invariants of the gradient: a single key gives dQ = dK = 0
    and dV = sum of dO; sum_j dK_j = 0; sum_j dV_j = sum_i dO_i; identical
    keys give dQ = 0; shifting every key by one vector changes nothing;
    linearity in dO; the last key of a causal square problem gets only the
    last query's gradient.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import backward as ob
from tiled_attention_10_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")

_TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def _raw16(x64: np.ndarray, dtype: str) -> torch.Tensor:
    """Round float64 values to the storage type (library conversion)."""
    return torch.from_numpy(x64).to(_TORCH_DT[dtype])


def _random_problem(B, H, H_kv, S_q, S_kv, D, dtype, layout, seed):
    g = np.random.default_rng(seed)
    shp = (lambda n, s: (B, n, s, D)) if layout == "BNSD" else (lambda n, s: (B, s, n, D))
    q = _raw16(g.standard_normal(shp(H, S_q)), dtype)
    k = _raw16(g.standard_normal(shp(H_kv, S_kv)), dtype)
    v = _raw16(g.standard_normal(shp(H_kv, S_kv)), dtype)
    do = _raw16(g.standard_normal(shp(H, S_q)), dtype)
    return q, k, v, do


def _bnsd64(x, layout):
    y = x.to(torch.float64)
    return y if layout == "BNSD" else y.permute(0, 2, 1, 3).contiguous()


def _torch_grads(q, k, v, do, layout, scale, causal, gqa):
    Q = _bnsd64(q, layout).requires_grad_()
    K = _bnsd64(k, layout).requires_grad_()
    V = _bnsd64(v, layout).requires_grad_()
    kw = {"enable_gqa": True} if gqa else {}
    O = F.scaled_dot_product_attention(Q, K, V, is_causal=causal, scale=scale, **kw)
    O.backward(_bnsd64(do, layout))
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


CASES = [
    # B, H, H_kv, S_q, S_kv, D, dtype, layout, causal, scale
    (1, 1, 1, 1, 1, 1, "bf16", "BNSD", False, 0.7),
    (2, 3, 3, 5, 7, 4, "bf16", "BNSD", False, 0.5),
    (2, 3, 3, 7, 5, 4, "f16", "BSND", True, 0.3),
    (1, 2, 2, 6, 6, 3, "f16", "BNSD", True, 1.1),
    (1, 4, 2, 9, 9, 8, "bf16", "BSND", True, 0.35),
    (2, 6, 2, 4, 11, 5, "f16", "BNSD", False, 0.9),
    (1, 2, 2, 40, 33, 16, "bf16", "BNSD", True, 0.25),
]


@pytest.mark.parametrize("B,H,H_kv,S_q,S_kv,D,dtype,layout,causal,scale", CASES)
def test_bwd_oracle_matches_torch_autograd(B, H, H_kv, S_q, S_kv, D, dtype, layout, causal, scale):
    # torch's is_causal is top-left aligned (query i sees keys j <= i), the
    # reading the forward oracle takes for S_q != S_kv as well.
    q, k, v, do = _random_problem(B, H, H_kv, S_q, S_kv, D, dtype, layout, seed=S_q * 31 + D)
    dQ, dK, dV = ob.attention_bwd(q, k, v, do, dtype=dtype, layout=layout, B=B, H=H, S_q=S_q,
                                  S_kv=S_kv, D=D, scale=scale, causal=causal, H_kv=H_kv)
    tq, tk, tv = _torch_grads(q, k, v, do, layout, scale, causal, gqa=H_kv != H)
    np.testing.assert_allclose(dQ, tq, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dK, tk, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dV, tv, rtol=1e-10, atol=1e-12)


def test_bwd_oracle_forward_matches_c_oracle():
    B, H, S_q, S_kv, D = 1, 2, 13, 17, 8
    q, k, v, do = _random_problem(B, H, H, S_q, S_kv, D, "bf16", "BNSD", seed=5)
    for causal in (False, True):
        O, lse = oracle.attention_full(q, k, v, dtype="bf16", layout="BNSD", B=B, H=H, S_q=S_q,
                                       S_kv=S_kv, D=D, scale=0.4, causal=causal)
        _, _, _, terms = ob.attention_bwd(q, k, v, do, dtype="bf16", layout="BNSD", B=B, H=H,
                                          S_q=S_q, S_kv=S_kv, D=D, scale=0.4, causal=causal,
                                          keep_terms=True)
        for h in range(H):
            np.testing.assert_allclose(terms[(0, h)]["O"], O[0, h], rtol=0, atol=1e-13)
            np.testing.assert_allclose(terms[(0, h)]["lse"], lse[0, h], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_oracle_matches_finite_differences(causal):
    # d/dx of L = sum(O * dO) by central differences of the forward, every
    # element of q, k and v of a small head.
    g = np.random.default_rng(11)
    S_q, S_kv, D, scale = 5, 6, 3, 0.8
    q, k, v, do = (g.standard_normal((S_q, D)), g.standard_normal((S_kv, D)),
                   g.standard_normal((S_kv, D)), g.standard_normal((S_q, D)))
    t = ob.head_terms(q, k, v, do, scale, causal)

    def loss(q_, k_, v_):
        return float((ob.head_terms(q_, k_, v_, do, scale, causal)["O"] * do).sum())

    eps = 1e-6
    for name, x, grad in (("q", q, t["dQ"]), ("k", k, t["dK"]), ("v", v, t["dV"])):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) -
                       loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * eps)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_single_key_closed_form():
    # One key: P = 1 everywhere, so dS = 0 (dQ = dK = 0) and dV = sum_i dO_i.
    g = np.random.default_rng(2)
    q, k, v, do = g.standard_normal((7, 4)), g.standard_normal((1, 4)), g.standard_normal((1, 4)), \
        g.standard_normal((7, 4))
    for causal in (False, True):
        t = ob.head_terms(q, k, v, do, 0.6, causal)
        np.testing.assert_allclose(t["dQ"], 0.0, atol=1e-15)
        np.testing.assert_allclose(t["dK"], 0.0, atol=1e-14)
        np.testing.assert_allclose(t["dV"][0], do.sum(axis=0), rtol=1e-14)


def test_two_keys_closed_form():
    # One query, two keys: P = (p, 1 - p) with p = sigmoid(scale q.(k0 - k1));
    # dS_0 = p (1 - p) (dO.(v0 - v1)) = -dS_1.
    q = np.array([[0.3, -1.2]])
    k = np.array([[0.5, 0.1], [-0.4, 0.9]])
    v = np.array([[1.0, 2.0], [-3.0, 0.5]])
    do = np.array([[0.7, -0.2]])
    scale = 0.9
    t = ob.head_terms(q, k, v, do, scale, False)
    p = 1.0 / (1.0 + np.exp(-scale * float(q[0] @ (k[0] - k[1]))))
    ds0 = p * (1 - p) * float(do[0] @ (v[0] - v[1]))
    np.testing.assert_allclose(t["dS"][0], [ds0, -ds0], rtol=1e-14)
    np.testing.assert_allclose(t["dQ"][0], scale * ds0 * (k[0] - k[1]), rtol=1e-13)
    np.testing.assert_allclose(t["dK"], scale * np.array([[ds0], [-ds0]]) * q, rtol=1e-13)
    np.testing.assert_allclose(t["dV"], np.array([[p], [1 - p]]) * do, rtol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sums(causal):
    # Rows of P sum to 1 and rows of dS sum to 0, so sum_j dK_j = 0 and
    # sum_j dV_j = sum_i dO_i.
    q, k, v, do = _random_problem(1, 2, 2, 19, 23, 6, "bf16", "BNSD", seed=3)
    dQ, dK, dV = ob.attention_bwd(q, k, v, do, dtype="bf16", layout="BNSD", B=1, H=2, S_q=19,
                                  S_kv=23, D=6, scale=0.5, causal=causal)
    np.testing.assert_allclose(dK.sum(axis=2), 0.0, atol=1e-12)
    dO64 = do.to(torch.float64).numpy()
    np.testing.assert_allclose(dV.sum(axis=2), dO64.sum(axis=2), rtol=1e-12, atol=1e-12)


def test_identical_keys_give_zero_dq():
    g = np.random.default_rng(4)
    q, v, do = g.standard_normal((9, 5)), g.standard_normal((12, 5)), g.standard_normal((9, 5))
    k = np.tile(g.standard_normal((1, 5)), (12, 1))
    for causal in (False, True):
        t = ob.head_terms(q, k, v, do, 0.7, causal)
        np.testing.assert_allclose(t["dQ"], 0.0, atol=1e-13)


def test_key_shift_invariance():
    # Adding one vector c to every key adds q.c to a whole row of S: P and
    # every gradient stay the same.
    g = np.random.default_rng(6)
    q, k, v, do = (g.standard_normal((8, 4)), g.standard_normal((10, 4)),
                   g.standard_normal((10, 4)), g.standard_normal((8, 4)))
    c = g.standard_normal((1, 4))
    for causal in (False, True):
        a = ob.head_terms(q, k, v, do, 0.5, causal)
        b = ob.head_terms(q, k + c, v, do, 0.5, causal)
        for name in ("dQ", "dK", "dV"):
            np.testing.assert_allclose(a[name], b[name], rtol=1e-11, atol=1e-12, err_msg=name)


def test_linearity_in_do():
    g = np.random.default_rng(8)
    q, k, v = g.standard_normal((6, 3)), g.standard_normal((7, 3)), g.standard_normal((7, 3))
    d1, d2 = g.standard_normal((6, 3)), g.standard_normal((6, 3))
    a, b = 0.75, -2.5
    t1 = ob.head_terms(q, k, v, d1, 0.9, True)
    t2 = ob.head_terms(q, k, v, d2, 0.9, True)
    t = ob.head_terms(q, k, v, a * d1 + b * d2, 0.9, True)
    for name in ("dQ", "dK", "dV"):
        np.testing.assert_allclose(t[name], a * t1[name] + b * t2[name], rtol=1e-12, atol=1e-13)


def test_causal_last_key_sees_only_last_query():
    # Square causal problem: key S-1 is visible to query S-1 alone.
    g = np.random.default_rng(9)
    S, D = 11, 4
    q, k, v, do = (g.standard_normal((S, D)) for _ in range(4))
    t = ob.head_terms(q, k, v, do, 0.6, True)
    np.testing.assert_allclose(t["dV"][-1], t["P"][-1, -1] * do[-1], rtol=1e-13)
    np.testing.assert_allclose(t["dK"][-1], 0.6 * t["dS"][-1, -1] * q[-1], rtol=1e-12)
    assert np.all(t["P"][np.triu_indices(S, 1)] == 0.0)


def test_gqa_gradient_is_sum_over_group():
    # A K/V head shared by g query heads gets the sum of the g per-head
    # gradients: compare with the same problem where K/V are repeated.
    q, k, v, do = _random_problem(1, 4, 2, 10, 12, 4, "bf16", "BNSD", seed=12)
    dQ, dK, dV = ob.attention_bwd(q, k, v, do, dtype="bf16", layout="BNSD", B=1, H=4, S_q=10,
                                  S_kv=12, D=4, scale=0.5, causal=True, H_kv=2)
    kr, vr = k.repeat_interleave(2, dim=1), v.repeat_interleave(2, dim=1)
    rQ, rK, rV = ob.attention_bwd(q, kr, vr, do, dtype="bf16", layout="BNSD", B=1, H=4, S_q=10,
                                  S_kv=12, D=4, scale=0.5, causal=True)
    np.testing.assert_allclose(dQ, rQ, rtol=1e-13)
    np.testing.assert_allclose(dK, rK.reshape(1, 2, 2, 12, 4).sum(axis=2), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dV, rV.reshape(1, 2, 2, 12, 4).sum(axis=2), rtol=1e-12, atol=1e-14)


def test_kv_head_subset_matches_full():
    w = Workload("t", 2, 4, 33, 40, 16, "bf16", "BSND", True, seed=1, H_kv=2)
    x = make_inputs(w)
    do = make_inputs(Workload("t", 2, 4, 33, 40, 16, "bf16", "BSND", True, seed=9)).q
    full = ob.attention_bwd(x.q, x.k, x.v, do, dtype="bf16", layout="BSND", B=2, H=4, S_q=33,
                            S_kv=40, D=16, scale=0.25, causal=True, H_kv=2)
    sub = ob.attention_bwd(x.q, x.k, x.v, do, dtype="bf16", layout="BSND", B=2, H=4, S_q=33,
                           S_kv=40, D=16, scale=0.25, causal=True, H_kv=2, kv_heads=[(1, 1)])
    np.testing.assert_array_equal(sub[0][1, 2:4], full[0][1, 2:4])
    np.testing.assert_array_equal(sub[1][1, 1], full[1][1, 1])
    np.testing.assert_array_equal(sub[2][1, 1], full[2][1, 1])
    assert np.isnan(sub[1][0]).all()
