"""ctypes binding of libfa_b200 (include/fa_api.h): argument marshalling only.

Every step of the forward pass runs in the CUDA library.  There is no CPU or
PyTorch fallback: if the library is missing, `load()` raises.
"""
from __future__ import annotations

import ctypes
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_b200.so")

FA_LAYOUT = {"BNSD": 0, "BSND": 1}
FA_DTYPE = {"f16": 0, "bf16": 1, "e4m3": 2}
FA_STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED",
             3: "FA_ERR_MISALIGNED", 4: "FA_ERR_CUDA", 5: "FA_ERR_DEVICE_TIMEOUT"}

# Symbols the header declares; the library must export all of them.
EXPORTS = ("fa_fwd", "fa_fwd_gqa", "fa_fwd_splitkv", "fa_fwd_splitkv_plan", "fa_fwd_splitkv_noalloc", "fa_bwd", "fa_bwd_workspace_size", "fa_fwd_varlen", "fa_fwd_paged", "fa_fwd_paged_split", "fa_fwd_paged_split_workspace_size", "fa_fwd_paged_split_plan", "fa_fwd_strided", "fa_bwd_strided", "fa_status_string", "fa_last_device_error", "fa_set_wait_limit_ns",
           "fa_probe_wait_timeout", "fa_version")



class Strides(ctypes.Structure):
    """fa_strides_t: element strides of a [B, H, S, D] tensor (D contiguous)."""
    _fields_ = [("batch", ctypes.c_int64), ("head", ctypes.c_int64), ("seq", ctypes.c_int64)]


def strides_of(t, order="BNSD"):
    """Strides of a torch tensor whose dims are [B, H, S, D] (order "BNSD") or
    [B, S, H, D] (order "BSND"); D must be contiguous."""
    st = t.stride()
    if st[3] != 1:
        raise ValueError("the head dimension must be contiguous")
    if order == "BNSD":
        return (st[0], st[1], st[2])
    return (st[0], st[2], st[1])


def _strides_array(triples):
    arr = (Strides * len(triples))()
    for i, (b, h, s_) in enumerate(triples):
        arr[i] = Strides(int(b), int(h), int(s_))
    return arr


_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {FA_STATUS.get(status, status)} ({fa_status_string(status)})")


def load(path: str = LIB_PATH):
    """Load libfa_b200.so (built by __graft_entry__.build()); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FileNotFoundError(
            f"{path} is missing: build the CUDA library first (python -c "
            "'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i64, f32, ip, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_uint64
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, f32, ip, ip, ip,
                           vp, vp, vp, vp]
    lib.fa_fwd.restype = ip
    lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, ip, ip, ip,
                               vp, vp, vp, vp]
    lib.fa_fwd_gqa.restype = ip
    sz = ctypes.c_size_t
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, ip, ip,
                                   ip, vp, vp, vp, ip, vp, sz, vp]
    lib.fa_fwd_splitkv.restype = ip
    lib.fa_fwd_splitkv_plan.argtypes = [i64, i64, i64, i64, i64, ctypes.POINTER(ip),
                                        ctypes.POINTER(sz)]
    lib.fa_fwd_splitkv_plan.restype = ip
    lib.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32,
                                           ip, ip, ip, vp, vp, vp, ip, vp]
    lib.fa_fwd_splitkv_noalloc.restype = ip
    lib.fa_bwd_workspace_size.argtypes = [i64, i64, i64, ctypes.POINTER(sz)]
    lib.fa_bwd_workspace_size.restype = ip
    lib.fa_bwd.argtypes = [vp] * 9 + [i64] * 6 + [f32, ip, ip, ip, vp, sz, vp]
    lib.fa_bwd.restype = ip
    lib.fa_fwd_varlen.argtypes = [vp] * 7 + [i64] * 7 + [f32, ip, ip, vp, vp, vp, vp]
    lib.fa_fwd_varlen.restype = ip
    lib.fa_fwd_paged.argtypes = [vp] * 8 + [i64] * 9 + [f32, ip, ip, vp, vp, vp, vp]
    lib.fa_fwd_paged.restype = ip
    lib.fa_fwd_strided.argtypes = [vp] * 5 + [i64] * 6 + [vp, f32, ip, ip, vp, vp, vp, vp]
    lib.fa_fwd_strided.restype = ip
    lib.fa_bwd_strided.argtypes = [vp] * 9 + [i64] * 6 + [vp, f32, ip, ip, vp, sz, vp]
    lib.fa_bwd_strided.restype = ip
    lib.fa_fwd_paged_split.argtypes = [vp] * 8 + [i64] * 9 + [f32, ip, ip, vp, vp, vp, ip, vp, sz,
                                                               vp]
    lib.fa_fwd_paged_split.restype = ip
    lib.fa_fwd_paged_split_workspace_size.argtypes = [i64, i64, i64, ip, i64, ctypes.POINTER(sz)]
    lib.fa_fwd_paged_split_workspace_size.restype = ip
    lib.fa_fwd_paged_split_plan.argtypes = [i64] * 8 + [ip, ctypes.POINTER(ip), ctypes.POINTER(sz)]
    lib.fa_fwd_paged_split_plan.restype = ip
    lib.fa_status_string.argtypes = [ip]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_last_device_error.argtypes = [vp]
    lib.fa_last_device_error.restype = ip
    lib.fa_set_wait_limit_ns.argtypes = [u64]
    lib.fa_set_wait_limit_ns.restype = None
    lib.fa_probe_wait_timeout.argtypes = [u64, vp]
    lib.fa_probe_wait_timeout.restype = ip
    lib.fa_version.argtypes = []
    lib.fa_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def fa_status_string(status: int) -> str:
    if _lib is None:
        return FA_STATUS.get(status, "unknown status")
    return _lib.fa_status_string(int(status)).decode()


def fa_fwd(q, k, v, o, lse, B, H, S_q, S_kv, D, scale, layout, causal, dtype,
           descale_q=None, descale_k=None, descale_v=None, stream=None) -> int:
    """Same arguments as the C call; pointers as ints (or None), enums as names
    or codes.  Returns the fa_status_t code."""
    lib = load()
    lay = FA_LAYOUT[layout] if isinstance(layout, str) else int(layout)
    dt = FA_DTYPE[dtype] if isinstance(dtype, str) else int(dtype)
    return int(lib.fa_fwd(q, k, v, o, lse, int(B), int(H), int(S_q), int(S_kv), int(D),
                          float(scale), lay, int(bool(causal)), dt, descale_q, descale_k,
                          descale_v, stream))


def fa_fwd_gqa(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, layout, causal, dtype,
               descale_q=None, descale_k=None, descale_v=None, stream=None) -> int:
    """Grouped-query variant: k and v have H_kv heads (query head h reads
    key/value head h // (H // H_kv)).  Returns the fa_status_t code."""
    lib = load()
    lay = FA_LAYOUT[layout] if isinstance(layout, str) else int(layout)
    dt = FA_DTYPE[dtype] if isinstance(dtype, str) else int(dtype)
    return int(lib.fa_fwd_gqa(q, k, v, o, lse, int(B), int(H), int(H_kv), int(S_q), int(S_kv),
                              int(D), float(scale), lay, int(bool(causal)), dt, descale_q,
                              descale_k, descale_v, stream))


def fa_fwd_splitkv_plan(B, H, S_q, S_kv, D):
    """(status, n_splits, workspace_bytes) chosen for the current device."""
    lib = load()
    n = ctypes.c_int(0)
    nb = ctypes.c_size_t(0)
    st = int(lib.fa_fwd_splitkv_plan(int(B), int(H), int(S_q), int(S_kv), int(D),
                                     ctypes.byref(n), ctypes.byref(nb)))
    return st, int(n.value), int(nb.value)


def fa_fwd_splitkv(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, layout, causal, dtype,
                   descale_q, descale_k, descale_v, n_splits, workspace, workspace_bytes,
                   stream=None) -> int:
    """Split-KV forward: partials in the caller's workspace, then the merge."""
    lib = load()
    lay = FA_LAYOUT[layout] if isinstance(layout, str) else int(layout)
    dt = FA_DTYPE[dtype] if isinstance(dtype, str) else int(dtype)
    return int(lib.fa_fwd_splitkv(q, k, v, o, lse, int(B), int(H), int(H_kv), int(S_q),
                                  int(S_kv), int(D), float(scale), lay, int(bool(causal)), dt,
                                  descale_q, descale_k, descale_v, int(n_splits), workspace,
                                  int(workspace_bytes), stream))


def fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, scale, layout, causal,
                           dtype, descale_q, descale_k, descale_v, n_splits, stream=None) -> int:
    """Split-KV forward with the library's fixed device scratch (no workspace
    argument, nothing allocated); FA_ERR_UNSUPPORTED when the partials need
    more than FA_NOALLOC_SCRATCH_BYTES."""
    lib = load()
    lay = FA_LAYOUT[layout] if isinstance(layout, str) else int(layout)
    dt = FA_DTYPE[dtype] if isinstance(dtype, str) else int(dtype)
    return int(lib.fa_fwd_splitkv_noalloc(q, k, v, o, lse, int(B), int(H), int(H_kv), int(S_q),
                                          int(S_kv), int(D), float(scale), lay,
                                          int(bool(causal)), dt, descale_q, descale_k, descale_v,
                                          int(n_splits), stream))


def fa_bwd_workspace_size(B, H, S_q):
    """(status, bytes) of device workspace fa_bwd needs."""
    lib = load()
    n = ctypes.c_size_t(0)
    st = int(lib.fa_bwd_workspace_size(int(B), int(H), int(S_q), ctypes.byref(n)))
    return st, int(n.value)


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S_q, S_kv, D, scale, layout, causal,
           dtype, workspace, workspace_bytes, stream=None) -> int:
    """Backward pass: dq, dk, dv from q, k, v, o, dout and lse (device pointers)."""
    lib = load()
    lay = FA_LAYOUT[layout] if isinstance(layout, str) else int(layout)
    dt = FA_DTYPE[dtype] if isinstance(dtype, str) else int(dtype)
    return int(lib.fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, int(B), int(H), int(H_kv), int(S_q),
                          int(S_kv), int(D), float(scale), lay, int(bool(causal)), dt, workspace,
                          int(workspace_bytes), stream))


CAUSAL = {"none": 0, "top_left": 1, "bottom_right": 2}


def fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, n_seqs, total_q, total_k, max_seqlen_q, H, H_kv,
                  D, scale, causal, dtype, descale_q=None, descale_k=None, descale_v=None,
                  stream=None) -> int:
    """Packed variable-length forward (device pointers; causal 0 / 1 / 2)."""
    lib = load()
    dt = FA_DTYPE[dtype] if isinstance(dtype, str) else int(dtype)
    c = CAUSAL[causal] if isinstance(causal, str) else int(causal)
    return int(lib.fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, int(n_seqs), int(total_q),
                                 int(total_k), int(max_seqlen_q), int(H), int(H_kv), int(D),
                                 float(scale), c, dt, descale_q, descale_k, descale_v, stream))


def fa_fwd_paged(q, k_cache, v_cache, o, lse, cu_q, seqused_k, block_table, n_seqs, max_pages,
                 page_size, num_pages, total_q, max_seqlen_q, H, H_kv, D, scale, causal, dtype,
                 descale_q=None, descale_k=None, descale_v=None, stream=None) -> int:
    """Packed queries against a paged K/V cache (device pointers)."""
    lib = load()
    dt = FA_DTYPE[dtype] if isinstance(dtype, str) else int(dtype)
    c = CAUSAL[causal] if isinstance(causal, str) else int(causal)
    return int(lib.fa_fwd_paged(q, k_cache, v_cache, o, lse, cu_q, seqused_k, block_table,
                                int(n_seqs), int(max_pages), int(page_size), int(num_pages),
                                int(total_q), int(max_seqlen_q), int(H), int(H_kv), int(D),
                                float(scale), c, dt, descale_q, descale_k, descale_v, stream))


def fa_fwd_paged_split_workspace_size(H, total_q, D, n_splits, n_seqs):
    """(status, bytes) of workspace fa_fwd_paged_split needs."""
    lib = load()
    n = ctypes.c_size_t(0)
    st = int(lib.fa_fwd_paged_split_workspace_size(int(H), int(total_q), int(D), int(n_splits),
                                                   int(n_seqs), ctypes.byref(n)))
    return st, int(n.value)


def fa_fwd_paged_split_plan(n_seqs, total_q, max_seqlen_q, total_k, max_seqlen_k, H, H_kv, D,
                            sm_count=0):
    """(status, n_splits, workspace bytes) for fa_fwd_paged_split; sm_count 0: this device."""
    lib = load()
    n = ctypes.c_int(0)
    b = ctypes.c_size_t(0)
    st = int(lib.fa_fwd_paged_split_plan(int(n_seqs), int(total_q), int(max_seqlen_q),
                                         int(total_k), int(max_seqlen_k), int(H), int(H_kv),
                                         int(D), int(sm_count), ctypes.byref(n), ctypes.byref(b)))
    return st, int(n.value), int(b.value)


def fa_fwd_paged_split(q, k_cache, v_cache, o, lse, cu_q, seqused_k, block_table, n_seqs,
                       max_pages, page_size, num_pages, total_q, max_seqlen_q, H, H_kv, D, scale,
                       causal, dtype, descale_q, descale_k, descale_v, n_splits, workspace,
                       workspace_bytes, stream=None) -> int:
    """Paged K/V forward with the keys split n_splits ways and merged."""
    lib = load()
    dt = FA_DTYPE[dtype] if isinstance(dtype, str) else int(dtype)
    c = CAUSAL[causal] if isinstance(causal, str) else int(causal)
    return int(lib.fa_fwd_paged_split(q, k_cache, v_cache, o, lse, cu_q, seqused_k, block_table,
                                      int(n_seqs), int(max_pages), int(page_size),
                                      int(num_pages), int(total_q), int(max_seqlen_q), int(H),
                                      int(H_kv), int(D), float(scale), c, dt, descale_q,
                                      descale_k, descale_v, int(n_splits), workspace,
                                      int(workspace_bytes), stream))


def fa_fwd_strided(q, k, v, o, lse, B, H, H_kv, S_q, S_kv, D, strides, scale, causal, dtype,
                   descale_q=None, descale_k=None, descale_v=None, stream=None) -> int:
    """Forward with explicit strides: `strides` = four (batch, head, seq) element
    triples for q, k, v, o (e.g. from strides_of)."""
    lib = load()
    dt = FA_DTYPE[dtype] if isinstance(dtype, str) else int(dtype)
    arr = None if strides is None else _strides_array(strides)
    return int(lib.fa_fwd_strided(q, k, v, o, lse, int(B), int(H), int(H_kv), int(S_q), int(S_kv),
                                  int(D), arr, float(scale), int(bool(causal)), dt, descale_q,
                                  descale_k, descale_v, stream))


def fa_bwd_strided(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S_q, S_kv, D, strides, scale,
                   causal, dtype, workspace, workspace_bytes, stream=None) -> int:
    """Backward with explicit strides: eight (batch, head, seq) triples for q, k,
    v, o, dout, dq, dk, dv."""
    lib = load()
    dt = FA_DTYPE[dtype] if isinstance(dtype, str) else int(dtype)
    arr = None if strides is None else _strides_array(strides)
    return int(lib.fa_bwd_strided(q, k, v, o, dout, lse, dq, dk, dv, int(B), int(H), int(H_kv),
                                  int(S_q), int(S_kv), int(D), arr, float(scale),
                                  int(bool(causal)), dt, workspace, int(workspace_bytes), stream))


def fa_last_device_error(stream=None) -> int:
    return int(load().fa_last_device_error(stream))


def fa_set_wait_limit_ns(ns: int) -> None:
    load().fa_set_wait_limit_ns(int(ns))


def fa_probe_wait_timeout(limit_ns: int, stream=None) -> int:
    return int(load().fa_probe_wait_timeout(int(limit_ns), stream))


# --------------------------------------------------------------------------
# Convenience wrapper over torch CUDA tensors (allocation only; the work is
# the single fa_fwd call).
# --------------------------------------------------------------------------
def attention(q, k, v, *, causal=False, scale=None, layout="BNSD", descale=None,
              out=None, lse=None, stream=None):
    """O, lse = attention(q, k, v): q/k/v torch CUDA tensors in `layout`
    (k and v may have fewer heads than q: grouped-query attention).

    dtype follows q (float16, bfloat16 or float8_e4m3fn).  `descale` for FP8 is
    a tuple of three 1-element fp32 CUDA tensors (or None for 1.0 each).
    """
    import torch
    dmap = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float8_e4m3fn: "e4m3"}
    if q.dtype not in dmap:
        raise TypeError(f"unsupported dtype {q.dtype}")
    dtype = dmap[q.dtype]
    if layout == "BNSD":
        B, H, S_q, D = q.shape
        H_kv, S_kv = k.shape[1], k.shape[2]
    else:
        B, S_q, H, D = q.shape
        S_kv, H_kv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    odt = torch.float16 if dtype == "f16" else torch.bfloat16
    if out is None:
        out = torch.empty(q.shape, dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S_q), dtype=torch.float32, device=q.device)
    ds = [None, None, None]
    if descale is not None:
        ds = [None if t is None else t.data_ptr() for t in descale]
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    st = fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B,
                    H, H_kv, S_q, S_kv, D, scale, layout, causal, dtype, ds[0], ds[1], ds[2],
                    stream)
    if st != 0:
        raise FaError(st, "fa_fwd")
    return out, lse


def attention_backward(q, k, v, out, lse, dout, *, causal=False, scale=None, layout="BNSD",
                       dq=None, dk=None, dv=None, stream=None):
    """dq, dk, dv = attention_backward(...): gradients through fa_bwd_strided
    for torch CUDA tensors in `layout` ([B, H, S, D] or [B, S, H, D] dims,
    any strides with D contiguous); `out`, `lse` from attention()."""
    import torch
    dmap = {torch.float16: "f16", torch.bfloat16: "bf16"}
    if q.dtype not in dmap:
        raise TypeError(f"no backward for {q.dtype}")
    dtype = dmap[q.dtype]
    if layout == "BNSD":
        B, H, S_q, D = q.shape
        H_kv, S_kv = k.shape[1], k.shape[2]
    else:
        B, S_q, H, D = q.shape
        S_kv, H_kv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q, memory_format=torch.contiguous_format) if dq is None else dq
    dk = torch.empty_like(k, memory_format=torch.contiguous_format) if dk is None else dk
    dv = torch.empty_like(v, memory_format=torch.contiguous_format) if dv is None else dv
    st, nbytes = fa_bwd_workspace_size(B, H, S_q)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    strides = [strides_of(t, layout) for t in (q, k, v, out, dout, dq, dk, dv)]
    st = fa_bwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), dout.data_ptr(),
                        lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, H_kv,
                        S_q, S_kv, D, strides, scale, causal, dtype, ws.data_ptr(), ws.numel(),
                        stream)
    if st != 0:
        raise FaError(st, "fa_bwd_strided")
    return dq, dk, dv


def _autograd_function():
    import torch

    class FlashAttention(torch.autograd.Function):
        """Autograd wrapper: forward through fa_fwd_strided, backward through
        fa_bwd_strided (fp16 / bf16)."""

        @staticmethod
        def forward(ctx, q, k, v, causal, scale, layout):
            if layout == "BNSD":
                B, H, S_q, D = q.shape
                H_kv, S_kv = k.shape[1], k.shape[2]
            else:
                B, S_q, H, D = q.shape
                S_kv, H_kv = k.shape[1], k.shape[2]
            sc = 1.0 / math.sqrt(D) if scale is None else scale
            out = torch.empty_like(q, memory_format=torch.contiguous_format)
            lse = torch.empty((B, H, S_q), dtype=torch.float32, device=q.device)
            dt = {torch.float16: "f16", torch.bfloat16: "bf16"}[q.dtype]
            stream = torch.cuda.current_stream(q.device).cuda_stream
            st = fa_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), B, H, H_kv, S_q, S_kv, D,
                                [strides_of(t, layout) for t in (q, k, v, out)], sc, causal, dt,
                                None, None, None, stream)
            if st != 0:
                raise FaError(st, "fa_fwd_strided")
            ctx.save_for_backward(q, k, v, out, lse)
            ctx.causal, ctx.scale, ctx.layout = causal, sc, layout
            return out

        @staticmethod
        def backward(ctx, dout):
            q, k, v, out, lse = ctx.saved_tensors
            if dout.stride(-1) != 1:
                dout = dout.contiguous()
            dq, dk, dv = attention_backward(q, k, v, out, lse, dout, causal=ctx.causal,
                                            scale=ctx.scale, layout=ctx.layout)
            return dq, dk, dv, None, None, None

    return FlashAttention


_FLASH_FN = None


def flash_attention(q, k, v, causal=False, scale=None, layout="BNSD"):
    """Differentiable attention (torch.autograd): O = softmax(scale q k^T) v
    with this library's forward and backward kernels (fp16 / bf16; k and v may
    have fewer heads than q; any strides with the head dim contiguous)."""
    global _FLASH_FN
    if _FLASH_FN is None:
        _FLASH_FN = _autograd_function()
    return _FLASH_FN.apply(q, k, v, causal, scale, layout)
