"""float64 CPU oracle for the FlashAttention forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``tiled_attention_10_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``fa_oracle.c`` (plain C, float64, OpenMP over rows or
heads); this module only compiles it with gcc and marshals numpy arrays into
it.  The definition it follows is the reference attention of the Ascend
FlashAttention page ("ops-transformer FlashAttention build and tuning",
section 4.3): softmax(scale * Q K^T, causal -inf above the diagonal) V, plus the
per-row natural-log log-sum-exp.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB = os.path.join(_HERE, "libfa_oracle.so")

DTYPE_CODES = {"f16": 0, "bf16": 1, "e4m3": 2}
LAYOUT_CODES = {"BNSD": 0, "BSND": 1}

_lib = None


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into libfa_oracle.so beside it (gcc, -O2, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # no OpenMP available
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, dbl, vp, ip = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        lib.fa_oracle_decode.argtypes = [vp, ip, i64, vp]
        lib.fa_oracle_rows.argtypes = [vp, vp, vp, ip, ip, i64, i64, i64, i64, i64,
                                       dbl, ip, dbl, dbl, dbl, i64, vp, vp, vp, vp, ip]
        lib.fa_oracle_full.argtypes = [vp, vp, vp, ip, ip, i64, i64, i64, i64, i64,
                                       dbl, ip, dbl, dbl, dbl, vp, vp, ip]
        lib.fa_oracle_rows_gqa.argtypes = [vp, vp, vp, ip, ip, i64, i64, i64, i64, i64, i64,
                                           dbl, ip, dbl, dbl, dbl, i64, vp, vp, vp, vp, ip]
        lib.fa_oracle_full_gqa.argtypes = [vp, vp, vp, ip, ip, i64, i64, i64, i64, i64, i64,
                                           dbl, ip, dbl, dbl, dbl, vp, vp, ip]
        lib.fa_oracle_max_threads.argtypes = []
        for f in (lib.fa_oracle_decode, lib.fa_oracle_rows, lib.fa_oracle_full,
                  lib.fa_oracle_rows_gqa, lib.fa_oracle_full_gqa, lib.fa_oracle_max_threads):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().fa_oracle_max_threads())


def _raw(x) -> np.ndarray:
    """Raw element bytes as a contiguous numpy array (accepts torch CPU tensors)."""
    if hasattr(x, "detach"):  # torch tensor: reinterpret its bytes, no value conversion
        import torch
        t = x.detach().contiguous().cpu()
        width = t.element_size()
        t = t.view(torch.uint8 if width == 1 else torch.int16)
        return t.numpy()
    return np.ascontiguousarray(x)


def decode(x, dtype: str) -> np.ndarray:
    """Decode raw f16 / bf16 / e4m3 elements to float64 with the oracle's decoder."""
    a = _raw(x)
    out = np.empty(a.size, dtype=np.float64)
    rc = _load().fa_oracle_decode(a.ctypes.data, DTYPE_CODES[dtype], a.size, out.ctypes.data)
    if rc:
        raise ValueError(f"fa_oracle_decode failed ({rc})")
    return out.reshape(a.shape)


def attention_rows(q, k, v, *, dtype, layout, B, H, S_q, S_kv, D, scale, causal,
                   rows, descale=(1.0, 1.0, 1.0), want_p=False, threads=0, H_kv=None):
    """Oracle output for selected rows.

    rows: int64 array [n, 3] of (b, h, i).  Returns (O [n, D], lse [n]) and,
    with want_p, P [n, S_kv].  Inputs are raw buffers in the given layout;
    K and V have H_kv heads (default H; query head h reads head h // (H // H_kv)).
    """
    qa, ka, va = _raw(q), _raw(k), _raw(v)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = r.shape[0]
    O = np.empty((n, D), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    P = np.empty((n, S_kv), dtype=np.float64) if want_p else None
    rc = _load().fa_oracle_rows_gqa(qa.ctypes.data, ka.ctypes.data, va.ctypes.data,
                                DTYPE_CODES[dtype], LAYOUT_CODES[layout], B, H,
                                H if H_kv is None else H_kv, S_q, S_kv, D,
                                float(scale), int(bool(causal)), float(descale[0]),
                                float(descale[1]), float(descale[2]), n, r.ctypes.data,
                                O.ctypes.data, lse.ctypes.data,
                                P.ctypes.data if want_p else None, int(threads))
    if rc:
        raise ValueError(f"fa_oracle_rows failed ({rc})")
    return (O, lse, P) if want_p else (O, lse)


def attention_full(q, k, v, *, dtype, layout, B, H, S_q, S_kv, D, scale, causal,
                   descale=(1.0, 1.0, 1.0), threads=0, H_kv=None):
    """Oracle output for every row: O [B, H, S_q, D] (BNSD order), lse [B, H, S_q].
    K and V have H_kv heads (default H)."""
    qa, ka, va = _raw(q), _raw(k), _raw(v)
    O = np.empty((B, H, S_q, D), dtype=np.float64)
    lse = np.empty((B, H, S_q), dtype=np.float64)
    rc = _load().fa_oracle_full_gqa(qa.ctypes.data, ka.ctypes.data, va.ctypes.data,
                                DTYPE_CODES[dtype], LAYOUT_CODES[layout], B, H,
                                H if H_kv is None else H_kv, S_q, S_kv, D,
                                float(scale), int(bool(causal)), float(descale[0]),
                                float(descale[1]), float(descale[2]), O.ctypes.data,
                                lse.ctypes.data, int(threads))
    if rc:
        raise ValueError(f"fa_oracle_full failed ({rc})")
    return O, lse
