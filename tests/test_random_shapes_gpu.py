"""Seeded random shapes: forward and every backward variant against the fp64 oracle.

Ten shapes drawn once from a fixed seed (odd sequence lengths from 1 to 700, every
head dim, both masks, scales from 0.02 to 0.3), so the ragged tails and tile counts
differ from the hand-picked cases elsewhere.  Tolerances as in the other parity tests.
Inputs have standard deviation 0.5, which keeps |O| below 2, where the spacing of bf16
values (at most 2^-8) is far below the 1e-2 bound on O; with unit inputs, sharp scales
and d = 256, |O| reaches 4-8, where storing O in bf16 alone can be off by 1.6e-2.
"""

import numpy as np
import pytest

import oracle
from tiled_attention_tmem_gb300 import binding as b, inputs as I

from helpers import check_fwd, check_grads, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _shapes():
    rng = np.random.default_rng(20261203)
    out = []
    for k in range(10):
        d = int(rng.choice([64, 96, 128, 192, 256]))
        B = int(rng.integers(1, 3))
        H = int(rng.integers(1, 4))
        N = int(rng.integers(1, 701))
        causal = bool(rng.integers(0, 2))
        scale = float(rng.uniform(0.02, 0.3))
        out.append((B, H, N, d, causal, scale, 3000 + k))
    return out


def _shapes_384():
    """Three more draws at head dim 384 (a seed of their own, so the set above stays)."""
    rng = np.random.default_rng(20261204)
    return [(int(rng.integers(1, 3)), int(rng.integers(1, 3)), int(rng.integers(1, 701)), 384,
             bool(rng.integers(0, 2)), float(rng.uniform(0.02, 0.1)), 3100 + k) for k in range(3)]


SHAPES = _shapes() + _shapes_384()


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}h{}n{}d{}{}".format(*s[:4], "c" if s[4] else ""))
def test_random_shape(shape):
    from tiled_attention_tmem_gb300 import api
    B, H, N, d, causal, scale, seed = shape
    x = I.make_inputs(B, H, N, d, seed=seed, sigma=0.5)
    q, k, v, do = (to_dev(t) for t in (x.q, x.k, x.v, x.do))
    o, lse = api.attention_forward(q, k, v, scale, causal)
    api.check_device_error()
    qf, kf, vf, dof = x.as_f64()
    o_ref, lse_ref = oracle.forward(qf, kf, vf, scale, causal)
    check_fwd(to_f64(o), to_f64(lse), o_ref, lse_ref, f"{shape}")
    ref = oracle.backward(qf, kf, vf, dof, scale, causal)
    for variant in (b.FA_BWD_5GEMM, b.FA_BWD_7GEMM):
        if b.lib().fa_bwd_launches(B, H, N, d, variant, int(causal)) == 0:
            continue
        grads = api.attention_backward(q, k, v, o, do, lse, scale, causal, variant=variant)
        api.check_device_error()
        check_grads([to_f64(g) for g in grads], ref, f"{shape} v{variant}")
