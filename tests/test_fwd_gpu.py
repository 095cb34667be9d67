"""Forward parity: the CUDA kernel (through the C ABI) against the fp64 CPU oracle."""

import numpy as np
import pytest

import oracle
from tiled_attention_tmem_gb300 import inputs as I

from helpers import check_fwd, head_f64, to_dev, to_f64

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
    # head dim 384 (Q in shared memory, S double-buffered next to a 384-column O):
    # one row, ragged tails, several tiles, both masks
    (1, 1, 1, 384, False, 1.0, 0.0, None),
    (1, 2, 1, 384, True, 1.0, 0.0, None),
    (1, 1, 129, 384, False, 1.0, 0.0, None),
    (1, 2, 129, 384, True, 1.0, 0.0, None),
    (1, 1, 1024, 384, False, 1.0, 0.0, None),
    (1, 1, 1024, 384, True, 1.0, 0.0, None),
    (2, 1, 333, 384, True, 0.5, 3.0, 1.0 / 20),
    # more work items than SMs, so that each persistent CTA runs several items,
    # short ones (one or two key tiles) among them
    (2, 96, 256, 256, True, 0.5, 0.0, 1.0 / 16),
    (1, 160, 130, 384, True, 0.5, 0.0, None),
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


def _lse_normalisation_error(qh, kh, scale, causal, rows, lse_got):
    """max_i |sum_j exp(s_ij - LSE_i) - 1| over the given rows, in fp64, with the GPU's LSE.

    The log-sum-exp is defined by this sum being one; an LSE error e moves it to
    exp(-e), so an LSE within the 1e-3 bound keeps it within expm1(1e-3) ~ 1.0e-3.
    """
    s = scale * (qh[rows] @ kh.T)
    if causal:
        s = np.where(np.arange(kh.shape[0])[None, :] <= np.asarray(rows)[:, None], s, -np.inf)
    return float(np.max(np.abs(np.sum(np.exp(s - np.asarray(lse_got)[:, None]), axis=1) - 1.0)))


# Full-size workloads in the bench's launch configuration (fa_fwd on the whole
# [B, H, N, d] problem).  Every head is checked: all of its rows where the oracle's
# N x N scores fit (the N = 2048 and the d = 256 workloads), sampled rows computed
# row by row otherwise (the N = 8192 workload).
FULL_EVERY_ROW = [I.CAUSAL_2K, I.HDIM256_4K]


@pytest.mark.parametrize("w", FULL_EVERY_ROW, ids=lambda w: w.name)
def test_forward_full_size_every_head_every_row(w):
    x = I.workload_inputs(w)
    o, lse = _run_fwd(x, w.B, w.H, w.N, w.d, w.softmax_scale, w.causal)
    o64, l64 = to_f64(o), to_f64(lse)
    for b in range(w.B):
        for h in range(w.H):
            qf, kf, vf, _ = head_f64(x, b, h)
            o_ref, lse_ref = oracle.forward(qf, kf, vf, w.softmax_scale, w.causal)
            check_fwd(o64[b, h], l64[b, h], o_ref[0, 0], lse_ref[0, 0], f"{w.name} b{b} h{h}")


def test_forward_full_size_every_head_sampled_rows():
    """B=2, H=16, N=8192 with keys shifted by +3: every head on sampled rows."""
    w = I.KSHIFT_8K
    x = I.workload_inputs(w)
    o, lse = _run_fwd(x, w.B, w.H, w.N, w.d, w.softmax_scale, w.causal)
    o64, l64 = to_f64(o), to_f64(lse)
    rng = np.random.default_rng(w.seed)
    worst = 0.0
    for b in range(w.B):
        for h in range(w.H):
            rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, w.N - 1],
                                             rng.integers(0, w.N, size=41)]))
            qf, kf, vf, _ = head_f64(x, b, h)
            o_ref, lse_ref = oracle.forward_rows(qf, kf, vf, w.softmax_scale, w.causal, 0, 0, rows)
            check_fwd(o64[b, h, rows], l64[b, h, rows], o_ref, lse_ref, f"{w.name} b{b} h{h}")
            worst = max(worst, _lse_normalisation_error(qf[0, 0], kf[0, 0], w.softmax_scale, w.causal, rows,
                                                        l64[b, h, rows]))
    assert worst <= np.expm1(1e-3) + 1e-9, f"sum_j exp(s_ij - LSE_i) off by {worst:.3e}"
