"""GPU parity: the C-ABI call against the float64 oracle, element by element.

Small shapes span several 128-row tiles and ragged tails; every output row is
compared.  Tolerances are the max-abs bounds of the method's specification:
O within 4e-3 (fp16), 1.6e-2 (bf16), 6e-2 (fp8 e4m3); lse within 1e-3.
"""
import math

import pytest
import torch

from tiled_attention_10_gb300.inputs import Workload
from tests.gpu_helpers import run_small

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, S_q, S_kv
    (1, 1, 128, 128),
    (1, 2, 256, 256),
    (2, 1, 384, 512),
    (1, 1, 1, 1),
    (1, 1, 2, 3),
    (1, 3, 63, 64),
    (2, 2, 127, 129),
    (1, 2, 129, 127),
    (1, 1, 255, 257),
    (1, 1, 300, 700),
    (2, 1, 640, 200),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,S_q,S_kv", SHAPES)
def test_parity_bnsd(B, H, S_q, S_kv, D, dtype, causal, cuda_lib):
    w = Workload("t", B, H, S_q, S_kv, D, dtype, "BNSD", causal, seed=S_q * 7 + S_kv)
    run_small(w)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,S_q,S_kv", [(2, 3, 200, 200), (1, 4, 129, 300), (2, 2, 513, 257)])
def test_parity_bsnd_poisoned(B, H, S_q, S_kv, D, dtype, causal, cuda_lib):
    """BSND with NaN bit patterns in the memory after the last valid row."""
    w = Workload("t", B, H, S_q, S_kv, D, dtype, "BSND", causal, poison=True, seed=S_q + 3 * S_kv)
    run_small(w)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S_q,S_kv", [(128, 128), (200, 333), (1, 1), (512, 512)])
def test_parity_fp8(S_q, S_kv, causal, cuda_lib):
    w = Workload("t", 1, 3, S_q, S_kv, 128, "e4m3", "BNSD", causal, seed=S_q + S_kv)
    run_small(w)


@pytest.mark.parametrize("scale", [0.0, 0.02, 1.0])
def test_parity_scales(scale, cuda_lib):
    w = Workload("t", 1, 2, 200, 260, 128, "bf16", "BNSD", True, scale=scale, seed=4)
    run_small(w)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 64), ("e4m3", 128), ("bf16", 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_parity_negative_scale(dtype, D, causal, cuda_lib):
    """A negative scale: the definition holds for any real scale; the
    products then compute -Q K^T and the softmax works with |scale|."""
    w = Workload("t", 1, 3, 200, 333, D, dtype, "BSND", causal, scale=-1.0 / math.sqrt(D),
                 seed=11 + D)
    run_small(w)


def test_large_logits_stay_finite(cuda_lib):
    """The FP16 overflow trap of the Ascend page (section 6.2): logits far above
    ln(65504) must not overflow -- scale 8 on N(0,1) data, D=64: scores ~ +-300."""
    w = Workload("t", 1, 2, 256, 256, 64, "f16", "BNSD", False, scale=8.0, seed=5)
    run_small(w)


def test_many_units_persistent_schedule(cuda_lib):
    """More units than SMs: every CTA walks several units."""
    w = Workload("t", 4, 40, 256, 256, 64, "bf16", "BNSD", True, seed=6)
    run_small(w)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "e4m3"])
@pytest.mark.parametrize("layout", ["BNSD", "BSND"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,H_kv", [(4, 2), (8, 1), (6, 3), (4, 4)])
def test_parity_gqa(H, H_kv, causal, layout, dtype, cuda_lib):
    """Grouped-query attention: query head h reads key/value head h // (H // H_kv)."""
    D = 128 if dtype == "e4m3" else 64
    w = Workload("t", 2, H, 300, 257, D, dtype, layout, causal, seed=H * 7 + H_kv, H_kv=H_kv,
                 poison=(layout == "BSND"))
    run_small(w)


@pytest.mark.parametrize("B,H,H_kv,S_q,S_kv,causal,seed", [
    (1, 6, 6, 385, 562, True, 1024), (3, 4, 4, 751, 625, True, 1117),
    (2, 2, 2, 898, 7, False, 1068), (3, 4, 1, 153, 187, True, 1003)])
def test_fp8_rows_with_few_keys(B, H, H_kv, S_q, S_kv, causal, seed, cuda_lib):
    """e4m3 P rounds each weight by up to 2^-4; rows that see only a few keys
    (the first query tile under a causal mask, keys shorter than a block) get
    P's rounding residual added too.  These shapes reached |dO| 0.052-0.062
    without it; the bound here is well inside the 6e-2 tolerance."""
    w = Workload("t", B, H, S_q, S_kv, 128, "e4m3", "BNSD", causal, seed=seed, H_kv=H_kv)
    eo, el = run_small(w)
    assert eo <= 0.035, eo
