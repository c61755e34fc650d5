"""fa_fwd_splitkv_noalloc: the split-KV forward pass with its partials in the
library's fixed device scratch (a static __device__ buffer of
FA_NOALLOC_SCRATCH_BYTES) instead of a caller workspace.

The file is collected last, so in a whole-suite run the scratch is set up on
a device that has already run every other entry point; it must also pass
alone in a fresh process.  GPU cases call the C ABI twice in a row and
compare both results with fa_fwd_splitkv (caller workspace, same split count,
same inputs) within the parity tolerance, and with the float64 oracle.
The CPU case checks that a problem larger than the scratch is refused before
any CUDA call.
"""
import numpy as np
import pytest
import torch

from tiled_attention_10_gb300 import binding
from tiled_attention_10_gb300.inputs import OUT_DTYPE, Workload, make_inputs, shape_of
from tests.gpu_helpers import (CANARY16, CANARY32, GUARD, TOL_LSE, TOL_O, compare_full,
                               sampled_rows_check, to_device)

SCRATCH_BYTES = 64 * 1024 * 1024   # FA_NOALLOC_SCRATCH_BYTES in include/fa_api.h


def _workspace_bytes(n_splits, B, H, S_q, D):
    rows = n_splits * B * H * S_q
    return ((rows * D * 4 + 255) // 256) * 256 + ((rows * 4 + 255) // 256) * 256


class _Out:
    """O and lse with canaries after them, in the workload's layout."""

    def __init__(self, w):
        oshape = shape_of(w.layout, w.B, w.H, w.S_q, w.D)
        n_o = int(np.prod(oshape))
        self.w = w
        self.o_buf = torch.full((n_o + GUARD,), CANARY16, dtype=torch.int16, device="cuda")
        self.o = self.o_buf[:n_o].view(OUT_DTYPE[w.dtype]).view(oshape)
        n_l = w.B * w.H * w.S_q
        self.l_buf = torch.full((n_l + GUARD,), CANARY32, dtype=torch.int32, device="cuda")
        self.lse = self.l_buf[:n_l].view(torch.float32).view(w.B, w.H, w.S_q)

    def guards_intact(self):
        return bool((self.o_buf[self.o.numel():] == CANARY16).all()) and \
            bool((self.l_buf[self.lse.numel():] == CANARY32).all())

    def o_bnsd64(self):
        o = self.o.float().cpu().double()
        if self.w.layout == "BSND":
            o = o.permute(0, 2, 1, 3)
        return o.contiguous().numpy()


def _args(w, q, k, v, out, ds):
    return (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.o.data_ptr(), out.lse.data_ptr(),
            w.B, w.H, w.kv_heads, w.S_q, w.S_kv, w.D, w.softmax_scale, w.layout, w.causal,
            w.dtype, ds[0], ds[1], ds[2])


def _descales(w, descale):
    if w.dtype != "e4m3":
        return [], [None, None, None]
    keep = [torch.tensor([d], dtype=torch.float32, device="cuda") for d in descale]
    return keep, [t.data_ptr() for t in keep]


def _with_workspace(w, q, k, v, descale, n_splits):
    """The existing entry point, with a NaN-filled caller workspace."""
    keep, ds = _descales(w, descale)
    out = _Out(w)
    ws = torch.full((_workspace_bytes(n_splits, w.B, w.H, w.S_q, w.D) // 4 + 64,), float("nan"),
                    device="cuda")
    st = binding.fa_fwd_splitkv(*_args(w, q, k, v, out, ds), n_splits, ws.data_ptr(),
                                ws.numel() * 4)
    torch.cuda.synchronize()
    assert st == 0, binding.FA_STATUS.get(st)
    assert binding.fa_last_device_error() == 0
    return out


def _no_alloc_twice(w, q, k, v, descale, n_splits):
    """Two calls in a row through fa_fwd_splitkv_noalloc, each into fresh outputs."""
    keep, ds = _descales(w, descale)
    outs = []
    for _ in range(2):
        out = _Out(w)
        torch.cuda.synchronize()
        st = binding.fa_fwd_splitkv_noalloc(*_args(w, q, k, v, out, ds), n_splits)
        assert st == 0, binding.FA_STATUS.get(st)
        outs.append(out)
    torch.cuda.synchronize()
    assert binding.fa_last_device_error() == 0
    for out in outs:
        assert out.guards_intact(), "write past the end of O or lse"
    return outs


def _close(w, a, b):
    do = float((a.o.float() - b.o.float()).abs().max())
    dl = float((a.lse - b.lse).abs().max())
    assert do <= TOL_O[w.dtype] and dl <= TOL_LSE, (do, dl)
    return do, dl


CASES = [
    # (workload, n_splits): tails in both S_q and S_kv, causal, GQA, BSND, fp8
    (Workload("t", 1, 4, 300, 5000, 128, "bf16", "BNSD", False, seed=11), 7),
    (Workload("t", 2, 8, 129, 3001, 64, "f16", "BSND", True, seed=12, H_kv=2, poison=True), 4),
    (Workload("t", 1, 4, 200, 2500, 128, "e4m3", "BNSD", True, seed=13, H_kv=1), 5),
    (Workload("t", 1, 2, 64, 700, 128, "bf16", "BNSD", False, seed=14), 1),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(CASES)))
def test_no_alloc_matches_workspace_entry_and_oracle(case, cuda_lib):
    w, n_splits = CASES[case]
    assert _workspace_bytes(n_splits, w.B, w.H, w.S_q, w.D) <= SCRATCH_BYTES
    x = make_inputs(w)
    q, k, v = to_device(x)
    ref = _with_workspace(w, q, k, v, x.descale, n_splits)
    first, second = _no_alloc_twice(w, q, k, v, x.descale, n_splits)
    for out in (first, second):
        do, dl = _close(w, out, ref)
        eo, el, og, lg = compare_full(w, out, x)
        assert np.isfinite(og).all() and np.isfinite(lg).all()
        assert eo <= TOL_O[w.dtype] and el <= TOL_LSE, (eo, el)
        print(f"case {case}: vs workspace entry max|dO|={do:.3g} max|dlse|={dl:.3g}; "
              f"vs oracle max|dO|={eo:.3g} max|dlse|={el:.3g}")


@pytest.mark.gpu
def test_no_alloc_near_scratch_capacity(cuda_lib):
    # 2 splits x 65027 rows: 67,108,096 bytes of partials (O and lse, each
    # 256-byte aligned), 768 bytes short of the 64 MiB scratch.
    w = Workload("t", 1, 1, 65027, 256, 128, "bf16", "BNSD", False, seed=15)
    need = _workspace_bytes(2, w.B, w.H, w.S_q, w.D)
    assert SCRATCH_BYTES - 1024 <= need <= SCRATCH_BYTES
    x = make_inputs(w, device="cuda")
    ref = _with_workspace(w, x.q, x.k, x.v, x.descale, 2)
    first, second = _no_alloc_twice(w, x.q, x.k, x.v, x.descale, 2)
    rows = [(0, 0, i) for i in (0, 1, 127, 128, 32767, 65024, 65025, 65026)]
    for out in (first, second):
        _close(w, out, ref)
        eo, el = sampled_rows_check(w, out, x.q, x.k, x.v, x.descale, rows)
        assert eo <= TOL_O[w.dtype] and el <= TOL_LSE, (eo, el)
    # one row more needs 256 bytes past the scratch: refused, nothing written
    w2 = Workload("t", 1, 1, 65028, 256, 128, "bf16", "BNSD", False, seed=15)
    assert _workspace_bytes(2, 1, 1, 65028, 128) > SCRATCH_BYTES
    x2 = make_inputs(w2, device="cuda")
    out = _Out(w2)
    st = binding.fa_fwd_splitkv_noalloc(*_args(w2, x2.q, x2.k, x2.v, out, [None] * 3), 2)
    torch.cuda.synchronize()
    assert st == 2, binding.FA_STATUS.get(st)                      # FA_ERR_UNSUPPORTED
    assert bool((out.o_buf.view(torch.int16) == CANARY16).all())


def test_no_alloc_refuses_oversize_on_host(built_lib):
    # Fake pointers, never dereferenced: a problem whose partials exceed the
    # scratch fails before any CUDA call, so this runs without a GPU.
    base = (16, 32, 48, 64, 80, 1, 1, 1, 65028, 256, 128, 0.1, "BNSD", 0, "bf16", None, None, None)
    assert binding.fa_fwd_splitkv_noalloc(*base, 2) == 2          # 256 bytes over: unsupported
    big = (16, 32, 48, 64, 80, 1, 64, 8, 65536, 65536, 128, 0.1, "BNSD", 0, "bf16", None, None,
           None)
    assert binding.fa_fwd_splitkv_noalloc(*big, 8) == 2           # 17 GB of partials
    assert binding.fa_fwd_splitkv_noalloc(*base, 0) == 1          # n_splits < 1
