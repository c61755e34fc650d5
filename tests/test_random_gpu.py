"""Seeded random problems against the oracle, forward and backward.

The fixed parity cases are chosen by hand; these draw the shape from a seeded
generator -- batch, query heads and their key/value grouping, S_q and S_kv
anywhere in 1..700 (ragged tails, S_q != S_kv), D, element type, layout,
causal or not, NaN-poisoned tails, and a scale of either sign or near zero (for
e4m3 within twice the default 1/sqrt(D), see _draw) --
so that combinations nobody listed still meet the same bounds: every output
element against the float64 oracle (forward: the dtype's tolerance on O,
1e-3 on lse; backward: the elementwise bound of tests/bwd_helpers.py).
"""
import math

import numpy as np
import pytest

from tiled_attention_10_gb300.inputs import Workload
from tests.gpu_helpers import run_small
from tests.test_bwd_gpu import _run_case

pytestmark = pytest.mark.gpu


def _draw(seed: int, bwd: bool, e4m3: bool = False) -> Workload:
    g = np.random.default_rng(seed)
    D = int(g.choice([64, 128]))
    dtypes = ["f16", "bf16"] if (bwd or D == 64) else ["f16", "bf16", "e4m3"]
    dtype = str(g.choice(dtypes))
    if e4m3:
        D, dtype = 128, "e4m3"
    H_kv = int(g.integers(1, 4))
    H = H_kv * int(g.choice([1, 2, 3, 4]))
    B = int(g.integers(1, 3))
    S_q, S_kv = int(g.integers(1, 701)), int(g.integers(1, 701))
    causal = bool(g.integers(0, 2))
    layout = str(g.choice(["BNSD", "BSND"]))
    if g.integers(0, 2):
        scale = float(g.choice([1.0, -1.0])) / math.sqrt(D)
    else:
        scale = float(g.uniform(-0.3, 0.3))
    if dtype == "e4m3":
        # e4m3 P keeps three mantissa bits, so O's error grows with the spread of
        # the logits: on N(0,1) inputs the max |dO| measured 0.023 / 0.043 / 0.059 /
        # 0.062 at |scale| = 1 / 2 / 2.5 / 3 times 1/sqrt(D).  The 6e-2 bound is the
        # method's for its own workloads (the default scale); draw within 2x it.
        lim = 2.0 / math.sqrt(D)
        scale = max(-lim, min(lim, scale))
    poison = bool(g.integers(0, 2))
    return Workload("rand", B, H, S_q, S_kv, D, dtype, layout, causal, scale=scale, seed=seed,
                    H_kv=H_kv, poison=poison, bwd=bwd)


@pytest.mark.parametrize("seed", range(24))
def test_random_forward(seed, cuda_lib):
    run_small(_draw(1000 + seed, bwd=False))


@pytest.mark.parametrize("seed", range(12))
def test_random_backward(seed, cuda_lib):
    _run_case(_draw(2000 + seed, bwd=True))


@pytest.mark.parametrize("seed", range(16))
def test_random_forward_e4m3(seed, cuda_lib):
    run_small(_draw(3000 + seed, bwd=False, e4m3=True))
