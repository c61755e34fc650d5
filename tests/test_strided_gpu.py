"""Strided tensors (fa_fwd_strided, fa_bwd_strided).

The Hygon retrospective's backward defect 13 stepped V by K's row stride; it
hid in every test where K and V had equal strides.  Here K and V always
differ: Q, K, V are views of a fused [B, S, 3, H, D] projection, or K is BNSD
while V is BSND with padded rows, outputs land in padded or fused buffers.
Each strided call must give the bits of the dense call on contiguous copies
(the same kernels on the same values), and the small forward case is also
checked against the float64 oracle.  Padding between rows must stay
untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward as ob
from tiled_attention_10_gb300 import binding
from tiled_attention_10_gb300.binding import strides_of

pytestmark = pytest.mark.gpu

PAD = 0x7BAD


def _fused_qkv(B, S, H, D, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    qkv = torch.randn(B, S, 3, H, D, generator=g, device="cuda").to(dtype)
    return qkv, qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]          # BSND views


def _padded(B, S, H, D, dtype, pad=64):
    """A [B, S, H, D] view into rows of D + pad elements filled with PAD bits."""
    buf = torch.full((B, S, H, D + pad), PAD, dtype=torch.int16, device="cuda").view(dtype)
    return buf, buf[..., :D]


def _dense_fwd(q, k, v, B, H, H_kv, S_q, S_kv, D, causal, dtype):
    qc, kc, vc = (t.contiguous() for t in (q, k, v))                 # BSND contiguous
    o = torch.empty_like(qc)
    lse = torch.empty(B, H, S_q, device="cuda")
    st = binding.fa_fwd_gqa(qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), B, H, H_kv, S_q, S_kv, D, 1 / np.sqrt(D), "BSND",
                            causal, dtype, None, None, None)
    assert st == 0
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_fused_qkv_into_padded_output(causal, cuda_lib):
    B, S, H, D = 2, 333, 4, 128
    qkv, q, k, v = _fused_qkv(B, S, H, D, torch.bfloat16, 1)
    obuf, o = _padded(B, S, H, D, torch.bfloat16)
    lse = torch.empty(B, H, S, device="cuda")
    st = binding.fa_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), B, H, H, S, S, D,
                                [strides_of(t, "BSND") for t in (q, k, v, o)], 1 / np.sqrt(D),
                                causal, "bf16")
    torch.cuda.synchronize()
    assert st == 0 and binding.fa_last_device_error() == 0
    o_ref, l_ref = _dense_fwd(q, k, v, B, H, H, S, S, D, causal, "bf16")
    assert torch.equal(o.contiguous().view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse, l_ref)
    assert bool((obuf.view(torch.int16)[..., D:] == PAD).all())     # padding untouched
    # and against the oracle
    O, L = oracle.attention_full(q.contiguous().cpu(), k.contiguous().cpu(), v.contiguous().cpu(),
                                 dtype="bf16", layout="BSND", B=B, H=H, S_q=S, S_kv=S, D=D,
                                 scale=1 / np.sqrt(D), causal=causal)
    og = o.float().permute(0, 2, 1, 3).cpu().double().numpy()
    assert np.abs(og - O).max() <= 1.6e-2 and np.abs(lse.cpu().double().numpy() - L).max() <= 1e-3


def test_fwd_k_and_v_with_different_strides_gqa(cuda_lib):
    # K: BNSD contiguous; V: BSND with padded rows; Q: BSND view of a wider tensor.
    B, H, H_kv, S_q, S_kv, D = 2, 8, 2, 200, 517, 64
    g = torch.Generator(device="cuda").manual_seed(2)
    qw = torch.randn(B, S_q, H, D + 32, generator=g, device="cuda").half()
    q = qw[..., :D]
    k_bnsd = torch.randn(B, H_kv, S_kv, D, generator=g, device="cuda").half()
    vbuf = torch.randn(B, S_kv, H_kv, D + 64, generator=g, device="cuda").half()
    v = vbuf[..., :D]
    o = torch.empty(B, H, S_q, D, device="cuda", dtype=torch.half)      # BNSD output
    lse = torch.empty(B, H, S_q, device="cuda")
    strides = [strides_of(q, "BSND"), strides_of(k_bnsd, "BNSD"), strides_of(v, "BSND"),
               strides_of(o, "BNSD")]
    assert strides[1][2] != strides[2][2]                              # K and V row strides differ
    st = binding.fa_fwd_strided(q.data_ptr(), k_bnsd.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), B, H, H_kv, S_q, S_kv, D, strides,
                                1 / np.sqrt(D), True, "f16")
    torch.cuda.synchronize()
    assert st == 0 and binding.fa_last_device_error() == 0
    o_ref, l_ref = _dense_fwd(q, k_bnsd.permute(0, 2, 1, 3), v, B, H, H_kv, S_q, S_kv, D, True, "f16")
    assert torch.equal(o.permute(0, 2, 1, 3).contiguous().view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse, l_ref)


@pytest.mark.parametrize("causal,H_kv", [(True, 4), (False, 2)])
def test_bwd_fused_qkv_into_fused_grads(causal, H_kv, cuda_lib):
    # The usual training layout: q, k, v views of one [B, S, 3, H, D] projection
    # (k, v use the first H_kv heads of their slots), gradients written into one
    # [B, S, 3, H, D] buffer; O and dO in padded rows.
    B, S, H, D = 2, 300, 4, 128
    qkv, q, k, v = _fused_qkv(B, S, H, D, torch.bfloat16, 3)
    k, v = k[:, :, :H_kv], v[:, :, :H_kv]
    scale = 1 / np.sqrt(D)
    obuf, o = _padded(B, S, H, D, torch.bfloat16)
    lse = torch.empty(B, H, S, device="cuda")
    assert binding.fa_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), B, H, H_kv, S, S, D,
                                  [strides_of(t, "BSND") for t in (q, k, v, o)], scale, causal,
                                  "bf16") == 0
    g = torch.Generator(device="cuda").manual_seed(4)
    dobuf, do = _padded(B, S, H, D, torch.bfloat16, pad=128)
    do.copy_(torch.randn(B, S, H, D, generator=g, device="cuda").to(torch.bfloat16))
    dqkv = torch.full((B, S, 3, H, D), PAD, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    dq, dk, dv = dqkv[:, :, 0], dqkv[:, :, 1, :H_kv], dqkv[:, :, 2, :H_kv]
    st, nb = binding.fa_bwd_workspace_size(B, H, S)
    ws = torch.empty(nb // 4 + 64, device="cuda")
    strides = [strides_of(t, "BSND") for t in (q, k, v, o, do, dq, dk, dv)]
    assert binding.fa_bwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                  dv.data_ptr(), B, H, H_kv, S, S, D, strides, scale, causal,
                                  "bf16", ws.data_ptr(), nb) == 0
    torch.cuda.synchronize()
    assert binding.fa_last_device_error() == 0
    # dense reference on contiguous copies
    qc, kc, vc, oc, doc = (t.contiguous() for t in (q, k, v, o, do))
    rq, rk, rv = torch.empty_like(qc), torch.empty_like(kc), torch.empty_like(vc)
    assert binding.fa_bwd(qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), oc.data_ptr(),
                          doc.data_ptr(), lse.data_ptr(), rq.data_ptr(), rk.data_ptr(),
                          rv.data_ptr(), B, H, H_kv, S, S, D, scale, "BSND", causal, "bf16",
                          ws.data_ptr(), nb) == 0
    torch.cuda.synchronize()
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert torch.equal(got.contiguous().view(torch.int16), ref.view(torch.int16))
    # the unused head slots of the fused gradient buffer stay untouched
    raw = dqkv.view(torch.int16)
    assert bool((raw[:, :, 1:, H_kv:] == PAD).all())
    # and the gradients against the float64 oracle (relative RMS sanity bound)
    dQ, dK, dV = ob.attention_bwd(qc.cpu(), kc.cpu(), vc.cpu(), doc.cpu(), dtype="bf16",
                                  layout="BSND", B=B, H=H, S_q=S, S_kv=S, D=D, scale=scale,
                                  causal=causal, H_kv=H_kv)
    for got, ref in ((dq, dQ), (dk, dK), (dv, dV)):
        gg = got.float().permute(0, 2, 1, 3).cpu().double().numpy()
        assert np.linalg.norm(gg - ref) <= 2e-2 * np.linalg.norm(ref)


@pytest.mark.parametrize("layout", ["BNSD", "BSND"])
def test_autograd_function_matches_direct_calls(layout, cuda_lib):
    # flash_attention (torch.autograd) = fa_fwd_strided + fa_bwd_strided: its
    # output and gradients equal the direct calls' bits.
    from tiled_attention_10_gb300 import flash_attention
    B, H, H_kv, S, D = 2, 4, 2, 257, 64
    g = torch.Generator(device="cuda").manual_seed(5)
    shp = (lambda n: (B, n, S, D)) if layout == "BNSD" else (lambda n: (B, S, n, D))
    q = torch.randn(*shp(H), generator=g, device="cuda").half().requires_grad_()
    k = torch.randn(*shp(H_kv), generator=g, device="cuda").half().requires_grad_()
    v = torch.randn(*shp(H_kv), generator=g, device="cuda").half().requires_grad_()
    do = torch.randn(*shp(H), generator=g, device="cuda").half()
    out = flash_attention(q, k, v, causal=True, layout=layout)
    out.backward(do)
    o_ref, lse_ref = binding.attention(q.detach(), k.detach(), v.detach(), causal=True,
                                       layout=layout)
    assert torch.equal(out.detach().view(torch.int16), o_ref.view(torch.int16))
    dq, dk, dv = binding.attention_backward(q.detach(), k.detach(), v.detach(), o_ref, lse_ref,
                                            do, causal=True, layout=layout)
    for got, ref in ((q.grad, dq), (k.grad, dk), (v.grad, dv)):
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
