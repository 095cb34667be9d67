"""Size extremes through the C ABI against the fp64 CPU oracle.

Thousands of short heads (far more work items than SMs, so every persistent CTA walks a
long list of one- and two-tile items) and one head of 32768 rows (the longest sequence
tested: few, long items, the split forward and both backward splits), each checked on
sampled heads or rows."""

import numpy as np
import pytest

import oracle
from tiled_attention_tmem_gb300 import inputs as I

from helpers import GradCheck, check_fwd, head_f64, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _fwd_bwd(x, d, causal, variant, splits=1):
    from tiled_attention_tmem_gb300 import api
    q, k, v, do = (to_dev(t) for t in (x.q, x.k, x.v, x.do))
    scale = 1.0 / np.sqrt(d)
    o, lse = api.attention_forward(q, k, v, scale, causal, splits=splits)
    grads = api.attention_backward(q, k, v, o, do, lse, scale, causal, variant=variant)
    api.check_device_error()
    return to_f64(o), to_f64(lse), [to_f64(t) for t in grads]


@pytest.mark.parametrize("variant", [5, 7])
def test_many_short_heads(variant):
    B, H, N, d, causal = 16, 256, 96, 64, True  # 4096 heads of a ragged length
    x = I.make_inputs(B, H, N, d, seed=3700 + variant)
    o, lse, grads = _fwd_bwd(x, d, causal, variant)
    scale = 1.0 / np.sqrt(d)
    rng = np.random.default_rng(3701)
    heads = [(0, 0), (B - 1, H - 1)] + [(int(rng.integers(B)), int(rng.integers(H))) for _ in range(6)]
    chk = GradCheck(f"{B}x{H} heads v{variant}")
    for bb, hh in heads:
        qf, kf, vf, dof = head_f64(x, bb, hh)
        o_ref, lse_ref = oracle.forward(qf, kf, vf, scale, causal)
        check_fwd(o[bb, hh], lse[bb, hh], o_ref[0, 0], lse_ref[0, 0], f"head ({bb}, {hh})")
        ref = oracle.backward(qf, kf, vf, dof, scale, causal)
        chk.add([t[bb, hh] for t in grads], [r[0, 0] for r in ref])
    chk.check()


def test_longest_single_head():
    B, H, N, d, causal = 1, 1, 32768, 128, True
    x = I.make_inputs(B, H, N, d, seed=3800)
    scale = 1.0 / np.sqrt(d)
    qf, kf, vf, dof = head_f64(x, 0, 0)
    rng = np.random.default_rng(3801)
    edge = [0, 1, 127, 128, N // 2, N - 129, N - 2, N - 1]
    rows = np.unique(np.concatenate([edge, rng.integers(0, N, size=24)]))
    o_ref, lse_ref = oracle.forward_rows(qf, kf, vf, scale, causal, 0, 0, rows)
    qrows = np.unique(np.concatenate([edge, rng.integers(0, N, size=12)]))
    krows = np.unique(np.concatenate([edge, rng.integers(0, N, size=12)]))
    ref = oracle.backward_rows(qf, kf, vf, dof, scale, causal, 0, 0, qrows, krows)
    for variant, splits in ((5, None), (7, 1)):
        o, lse, g = _fwd_bwd(x, d, causal, variant, splits)
        check_fwd(o[0, 0, rows], lse[0, 0, rows], o_ref, lse_ref, f"N={N} fwd (splits {splits})")
        chk = GradCheck(f"N={N} v{variant}")
        chk.add((g[0][0, 0, qrows], g[1][0, 0, krows], g[2][0, 0, krows]), ref)
        chk.check()
