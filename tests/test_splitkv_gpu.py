"""Split-KV forward (fa_fwd_splitkv): parity with the float64 oracle for many
split counts, masks, tails, layouts, GQA and fp8, plus the argument checks.
The split run reaches the same attention, so the oracle is the plain one."""
import numpy as np
import pytest
import torch

from tiled_attention_10_gb300 import binding
from tiled_attention_10_gb300.inputs import OUT_DTYPE, Workload, make_inputs, shape_of
from tests.gpu_helpers import CANARY16, CANARY32, GUARD, TOL_LSE, TOL_O, compare_full, to_device

pytestmark = pytest.mark.gpu


class SplitRun:
    def __init__(self, w, q, k, v, descale, n_splits, ws_extra=0):
        dev = q.device
        oshape = shape_of(w.layout, w.B, w.H, w.S_q, w.D)
        n_o = int(np.prod(oshape))
        self.w = w
        self.o_buf = torch.full((n_o + GUARD,), CANARY16, dtype=torch.int16, device=dev)
        self.o = self.o_buf[:n_o].view(OUT_DTYPE[w.dtype]).view(oshape)
        n_l = w.B * w.H * w.S_q
        self.l_buf = torch.full((n_l + GUARD,), CANARY32, dtype=torch.int32, device=dev)
        self.lse = self.l_buf[:n_l].view(torch.float32).view(w.B, w.H, w.S_q)
        st, _, need = binding.fa_fwd_splitkv_plan(w.B, w.H, w.S_q, w.S_kv, w.D)
        assert st == 0
        rows = n_splits * w.B * w.H * w.S_q
        need = ((rows * w.D * 4 + 255) // 256) * 256 + ((rows * 4 + 255) // 256) * 256
        # NaN-filled workspace: nothing may read a partial that was not written
        self.ws = torch.full((need // 4 + 64 + ws_extra,), float("nan"), device=dev)
        ds = [None, None, None]
        if w.dtype == "e4m3":
            self._ds = [torch.tensor([d], dtype=torch.float32, device=dev) for d in descale]
            ds = [t.data_ptr() for t in self._ds]
        self.status = binding.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             self.o.data_ptr(), self.lse.data_ptr(), w.B, w.H,
                                             w.kv_heads, w.S_q, w.S_kv, w.D, w.softmax_scale,
                                             w.layout, w.causal, w.dtype, ds[0], ds[1], ds[2],
                                             n_splits, self.ws.data_ptr(), self.ws.numel() * 4)
        self.device_status = binding.fa_last_device_error()

    def guards_intact(self):
        return bool((self.o_buf[self.o.numel():] == CANARY16).all()) and \
            bool((self.l_buf[self.lse.numel():] == CANARY32).all())

    def o_bnsd64(self):
        o = self.o.float().cpu().double()
        if self.w.layout == "BSND":
            o = o.permute(0, 2, 1, 3)
        return o.contiguous().numpy()


def _run(w, n_splits):
    x = make_inputs(w)
    q, k, v = to_device(x)
    r = SplitRun(w, q, k, v, x.descale, n_splits)
    torch.cuda.synchronize()
    assert r.status == 0, binding.FA_STATUS.get(r.status)
    assert r.device_status == 0
    assert r.guards_intact()
    eo, el, og, lg = compare_full(w, r, x)
    assert np.isfinite(og).all() and np.isfinite(lg).all()
    assert eo <= TOL_O[w.dtype] and el <= TOL_LSE, (eo, el)
    return eo, el


@pytest.mark.parametrize("n_splits", [1, 2, 3, 5, 8, 32])
@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_parity_split_counts(n_splits, causal, cuda_lib):
    w = Workload("t", 1, 2, 300, 1100, 128, "bf16", "BNSD", causal, seed=n_splits)
    _run(w, n_splits)


@pytest.mark.parametrize("dtype", ["f16", "e4m3"])
@pytest.mark.parametrize("layout", ["BNSD", "BSND"])
def test_splitkv_parity_dtypes_layouts(dtype, layout, cuda_lib):
    D = 128 if dtype == "e4m3" else 64
    w = Workload("t", 2, 4, 129, 777, D, dtype, layout, True, seed=3, H_kv=2,
                 poison=(layout == "BSND"))
    _run(w, 4)


@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_negative_scale(causal, cuda_lib):
    """A negative scale through the split path and the merge."""
    w = Workload("t", 1, 4, 130, 1500, 128, "bf16", "BNSD", causal, scale=-0.3, seed=12)
    _run(w, 4)


def test_splitkv_more_splits_than_blocks(cuda_lib):
    """Splits beyond the key blocks are empty: zero weight, never read."""
    w = Workload("t", 1, 2, 200, 300, 128, "bf16", "BNSD", False, seed=4)
    _run(w, 7)


def test_splitkv_equals_whole_pass(cuda_lib):
    w = Workload("t", 2, 3, 257, 2000, 128, "bf16", "BSND", True, seed=5)
    x = make_inputs(w, device="cuda")
    a = SplitRun(w, x.q, x.k, x.v, x.descale, 1)
    b = SplitRun(w, x.q, x.k, x.v, x.descale, 6)
    torch.cuda.synchronize()
    assert a.status == 0 and b.status == 0
    assert float((a.o.float() - b.o.float()).abs().max()) <= 1.6e-2
    assert float((a.lse - b.lse).abs().max()) <= 1e-4


def test_splitkv_plan_and_argument_checks(cuda_lib):
    st, n, nb = binding.fa_fwd_splitkv_plan(1, 8, 512, 16384, 128)
    assert st == 0 and 1 < n <= 32 and nb > 0
    st, n, nb = binding.fa_fwd_splitkv_plan(4, 32, 4096, 4096, 128)
    assert st == 0 and n == 1 and nb == 0
    w = Workload("t", 1, 1, 128, 512, 128, "bf16", "BNSD", False, seed=6)
    x = make_inputs(w, device="cuda")
    o = torch.empty_like(x.q)
    lse = torch.empty(1, 1, 128, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    args = (x.q.data_ptr(), x.k.data_ptr(), x.v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1,
            1, 128, 512, 128, 0.1, "BNSD", False, "bf16", None, None, None)
    assert binding.fa_fwd_splitkv(*args, 0, ws.data_ptr(), ws.numel()) == 1
    assert binding.fa_fwd_splitkv(*args, 33, ws.data_ptr(), ws.numel()) == 2
    assert binding.fa_fwd_splitkv(*args, 4, ws.data_ptr(), 100) == 1
    assert binding.fa_fwd_splitkv(*args, 4, None, ws.numel()) == 1
    assert binding.fa_fwd_splitkv(*args, 4, ws.data_ptr() + 16, ws.numel() - 16) == 3


def test_splitkv_workload_full_size(cuda_lib):
    """The measured split workload (8 heads, 512 queries, 16384 keys) with the
    planned split count, on sampled rows."""
    from tiled_attention_10_gb300.inputs import EXTRA_WORKLOADS, sample_rows
    from tests.gpu_helpers import sampled_rows_check
    w = EXTRA_WORKLOADS["bf16_splitkv_1x8x512x16384x128"]
    st, n, _ = binding.fa_fwd_splitkv_plan(w.B, w.H, w.S_q, w.S_kv, w.D)
    assert st == 0 and n > 1
    x = make_inputs(w, device="cuda")
    r = SplitRun(w, x.q, x.k, x.v, x.descale, n)
    torch.cuda.synchronize()
    assert r.status == 0 and r.device_status == 0 and r.guards_intact()
    assert bool(torch.isfinite(r.o.float()).all()) and bool(torch.isfinite(r.lse).all())
    rows = [tuple(int(v) for v in t) for t in sample_rows(w, 48, seed=3)]
    eo, el = sampled_rows_check(w, r, x.q, x.k, x.v, x.descale, rows)
    print(f"split workload (n_splits={n}): max|dO|={eo:.3g} max|dlse|={el:.3g}")
    assert eo <= TOL_O[w.dtype] and el <= TOL_LSE, (eo, el)
