"""The C-ABI library: it builds, loads, exports every symbol include/fa_api.h
declares, and rejects bad arguments on the host before touching a device.
No test here launches a kernel, so they all run without a GPU."""
import ctypes
import os
import re

import pytest

from tiled_attention_10_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib(built_lib):
    return built_lib


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "fa_api.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_what_binding_expects():
    assert set(_declared_functions()) == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(6):
        s = binding.fa_status_string(code)
        assert s and s != "unknown status"
    assert binding.fa_status_string(99) == "unknown status"
    assert lib.fa_version().decode().count(".") == 2


GOOD = dict(q=16, k=32, v=48, o=64, lse=80, B=1, H=1, S_q=8, S_kv=8, D=128, scale=0.1,
            layout="BNSD", causal=0, dtype="bf16")


def _call(**over):
    a = dict(GOOD)
    a.update(over)
    return binding.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["S_q"],
                          a["S_kv"], a["D"], a["scale"], a["layout"], a["causal"], a["dtype"],
                          a.get("dq"), a.get("dk"), a.get("dv"), None)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(o=None), 1), (dict(lse=None), 1),
    (dict(B=0), 1), (dict(H=0), 1), (dict(S_q=0), 1), (dict(S_kv=0), 1), (dict(D=0), 1),
    (dict(S_kv=-5), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(scale=float("-inf")), 1), (dict(layout=7), 1), (dict(dtype=9), 1),
    (dict(dq=16), 1),                                   # descale with a 16-bit dtype
    (dict(D=96), 2), (dict(D=256), 2), (dict(D=64, dtype="e4m3"), 2),
    (dict(S_q=1 << 31), 2),
    (dict(q=8), 3), (dict(o=24), 3), (dict(lse=82), 3),
    (dict(dtype="e4m3", dq=18), 3),
])
def test_invalid_arguments_rejected_on_host(lib, over, code):
    # Pointers are fake and never dereferenced: every case fails validation
    # before any CUDA call.
    assert _call(**over) == code


def test_loads_without_gpu_and_does_not_fallback():
    # The binding has no CPU path: the only compute entry point is the C call.
    src = open(os.path.join(ROOT, "tiled_attention_10_gb300", "binding.py")).read()
    assert "oracle" not in src
    assert "scaled_dot_product_attention" not in src


def _call_gqa(**over):
    a = dict(GOOD, H=4, H_kv=2)
    a.update(over)
    return binding.fa_fwd_gqa(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["H_kv"],
                              a["S_q"], a["S_kv"], a["D"], a["scale"], a["layout"], a["causal"],
                              a["dtype"], None, None, None, None)


@pytest.mark.parametrize("over,code", [
    (dict(H_kv=0), 1), (dict(H_kv=3), 1), (dict(H=4, H_kv=8), 1), (dict(q=None), 1),
    (dict(D=80), 2), (dict(k=40), 3),
])
def test_gqa_invalid_arguments_rejected_on_host(lib, over, code):
    assert _call_gqa(**over) == code


def test_splitkv_host_checks(lib):
    # fake pointers, never dereferenced: each case fails before any CUDA call
    base = (16, 32, 48, 64, 80, 1, 2, 2, 8, 512, 128, 0.1, "BNSD", 0, "bf16", None, None, None)
    assert binding.fa_fwd_splitkv(*base, 0, 4096, 1 << 20) == 1        # n_splits < 1
    assert binding.fa_fwd_splitkv(*base, 64, 4096, 1 << 20) == 2       # too many splits
    assert binding.fa_fwd_splitkv(*base, 4, None, 1 << 20) == 1        # no workspace
    assert binding.fa_fwd_splitkv(*base, 4, 4096, 8) == 1              # too small
    assert binding.fa_fwd_splitkv(*base, 4, 4112, 1 << 20) == 3        # not 256-aligned
    bad = (16, 32, 48, 64, 80, 1, 3, 2, 8, 512, 128, 0.1, "BNSD", 0, "bf16", None, None, None)
    assert binding.fa_fwd_splitkv(*bad, 4, 4096, 1 << 20) == 1         # H % H_kv != 0


def test_bwd_host_checks(lib):
    # fake pointers, never dereferenced: each case fails before any CUDA call
    st, n = binding.fa_bwd_workspace_size(2, 4, 300)
    assert st == 0 and n == 2 * ((2 * 4 * 384 * 4 + 255) // 256 * 256)
    assert binding.fa_bwd_workspace_size(0, 4, 300)[0] == 1
    p = [16 * (i + 1) for i in range(9)]
    base = p + [2, 4, 2, 300, 300, 128, 0.1, "BNSD", 1, "bf16"]
    assert binding.fa_bwd(*base, 4096, 8) == 1                      # workspace too small
    assert binding.fa_bwd(*base, None, n) == 1                      # no workspace
    assert binding.fa_bwd(*base, 4096 + 16, n) == 3                 # workspace off 256 bytes
    fp8 = p + [2, 4, 2, 300, 300, 128, 0.1, "BNSD", 1, "e4m3"]
    assert binding.fa_bwd(*fp8, 4096, n) == 2                       # no fp8 backward
    nodq = list(p)
    nodq[6] = None
    assert binding.fa_bwd(*(nodq + [2, 4, 2, 300, 300, 128, 0.1, "BNSD", 1, "bf16"]), 4096, n) == 1
    odd = list(p)
    odd[7] = 16 * 8 + 2
    assert binding.fa_bwd(*(odd + [2, 4, 2, 300, 300, 128, 0.1, "BNSD", 1, "bf16"]), 4096, n) == 3
    assert binding.fa_bwd(*(p + [2, 4, 3, 300, 300, 128, 0.1, "BNSD", 1, "bf16"]), 4096, n) == 1
    assert binding.fa_bwd(*(p + [2, 4, 2, 300, 300, 80, 0.1, "BNSD", 1, "bf16"]), 4096, n) == 2


def test_varlen_paged_host_checks(lib):
    # fake pointers, never dereferenced: each case fails before any CUDA call
    a = 4096
    vb = [a] * 7 + [2, 300, 300, 300, 4, 2, 128, 0.1, 1, "bf16"]
    assert binding.fa_fwd_varlen(*vb[:5], None, *vb[6:]) == 1          # no cu_seqlens_q
    assert binding.fa_fwd_varlen(*vb[:7], 0, *vb[8:]) == 1             # n_seqs < 1
    assert binding.fa_fwd_varlen(*vb[:16], 3, "bf16") == 1             # causal 3
    assert binding.fa_fwd_varlen(*vb[:13], 80, *vb[14:]) == 2          # D = 80
    assert binding.fa_fwd_varlen(*vb[:6], a + 2, *vb[7:]) == 3         # cu_seqlens_k off 4 bytes
    assert binding.fa_fwd_varlen(*vb[:8], 0, *vb[9:]) == 0             # total_q = 0: nothing to do
    pg = [a] * 8 + [2, 8, 64, 100, 300, 300, 4, 2, 128, 0.1, 2, "bf16"]
    assert binding.fa_fwd_paged(*pg[:10], 48, *pg[11:]) == 2           # page size 48
    assert binding.fa_fwd_paged(*pg[:10], 8, *pg[11:]) == 1            # page size < 16
    assert binding.fa_fwd_paged(*pg[:7], None, *pg[8:]) == 1           # no block table
    assert binding.fa_fwd_paged(*pg[:9], 0, *pg[10:]) == 1             # max pages 0
    assert binding.fa_fwd_paged(*pg[:15], 3, *pg[16:]) == 1            # H % H_kv != 0


def test_paged_split_workspace_size(lib):
    # the sequence order (int32 per sequence, up to 16384 sequences) then, for
    # n_splits > 1, fp32 partial O and lse; each part rounded up to 256 bytes
    r = lambda n: -(-n // 256) * 256
    H, tq, D = 32, 128, 128
    assert binding.fa_fwd_paged_split_workspace_size(H, tq, D, 1, 128) == (0, r(128 * 4))
    assert binding.fa_fwd_paged_split_workspace_size(H, tq, D, 1, 1) == (0, 256)
    part = r(2 * H * tq * D * 4) + r(2 * H * tq * 4)
    assert binding.fa_fwd_paged_split_workspace_size(H, tq, D, 2, 128) == (0, r(512) + part)
    assert binding.fa_fwd_paged_split_workspace_size(H, tq, D, 1, 16384) == (0, 65536)
    assert binding.fa_fwd_paged_split_workspace_size(H, tq, D, 1, 16385) == (0, 0)   # given order
    assert binding.fa_fwd_paged_split_workspace_size(H, tq, D, 1, 0)[0] == 1
    assert binding.fa_fwd_paged_split_workspace_size(H, tq, D, 0, 4)[0] == 1
    # a workspace smaller than that is rejected before any CUDA call
    a = 4096
    ps = [a] * 8 + [4, 8, 64, 100, 4, 1, 32, 8, 128, 0.1, 2, "bf16", None, None, None]
    assert binding.fa_fwd_paged_split(*ps, 1, a, 255) == 1             # order needs 256
    assert binding.fa_fwd_paged_split(*ps, 2, None, 0) == 1            # n_splits > 1 needs one
    assert binding.fa_fwd_paged_split(*ps, 2, a + 16, 1 << 30) == 3    # workspace off 256 bytes


def test_paged_split_plan(lib):
    # host arithmetic only (sm_count given): decode over 1K-32K keys, 8 key/value
    # heads with 4 query heads each (one packed tile per sequence and head)
    plan = lambda n, tk, mk, sm=152, tq=None, mq=1, H=32, H_kv=8: binding.fa_fwd_paged_split_plan(
        n, n if tq is None else tq, mq, tk, mk, H, H_kv, 128, sm)
    # 128 sequences, 1.03M keys: a two-way split of the longest (255 blocks)
    # is within half an SM's share (428 blocks)
    st, n, ws = plan(128, 1033533, 32623)
    assert (st, n) == (0, 2)
    assert ws == binding.fa_fwd_paged_split_workspace_size(32, 128, 128, 2, 128)[1]
    # 32 sequences, 265K keys: share 110 blocks, longest 232 -> five ways
    assert plan(32, 265332, 29592)[:2] == (0, 5)
    # the same keys with 4x the SMs need more splits, never fewer
    ns = [plan(32, 265332, 29592, sm=sm)[1] for sm in (38, 76, 152, 304, 608)]
    assert ns == sorted(ns) and ns[-1] <= 32
    # a lone short sequence: at least two key blocks per split (8 blocks -> 4)
    assert plan(1, 1000, 1000)[:2] == (0, 4)
    assert plan(1, 128, 128)[:2] == (0, 1)
    # prefill that fills the GPU on its own: no split, and the workspace is
    # then the sequence order alone
    st, n, ws = plan(64, 64 * 8192, 8192, tq=64 * 4096, mq=4096)
    assert (st, n, ws) == (0, 1, 256)
    # the cap: 32 splits
    assert plan(1, 1 << 20, 1 << 20, sm=100000)[:2] == (0, 32)
    for bad in ((0, 10, 10), (4, 10, 11), (4, -1, 0)):
        assert plan(*bad)[0] == 1
    assert plan(4, 100, 10, H=32, H_kv=6)[0] == 1     # H % H_kv != 0
    assert plan(4, 100, 10, sm=-1)[0] == 1


def test_strided_host_checks(lib):
    # fake pointers, never dereferenced: each case fails before any CUDA call
    a = 4096
    good = [(4 * 8 * 64, 64, 8 * 64)] * 4           # BSND-like, bf16: all 16-byte multiples
    args = [a] * 5 + [2, 4, 4, 8, 8, 64]
    assert binding.fa_fwd_strided(*args, None, 0.1, 0, "bf16") == 1          # no strides
    assert binding.fa_fwd_strided(*args, good[:3] + [(0, 64, 512)], 0.1, 0, "bf16") == 1
    assert binding.fa_fwd_strided(*args, good[:3] + [(2052, 64, 512)], 0.1, 0, "bf16") == 3
    assert binding.fa_fwd_strided(*args, good[:3] + [(1 << 39, 64, 512)], 0.1, 0, "bf16") == 2
    bargs = [a] * 9 + [2, 4, 4, 8, 8, 64]
    assert binding.fa_bwd_strided(*bargs, good * 2, 0.1, 0, "bf16", None, 0) == 1  # no workspace
    assert binding.fa_bwd_strided(*bargs, good * 2, 0.1, 0, "e4m3", a, 1 << 20) == 2  # no fp8 backward
    bad = good * 2
    bad[7] = (2052, 64, 512)                                                  # dv batch stride: 4104 bytes
    assert binding.fa_bwd_strided(*bargs, bad, 0.1, 0, "bf16", a, 1 << 20) == 3
