"""Parity on the sequence sweep and the head-dim sweep, in the launch configuration
the bench measures (fa_fwd, then fa_bwd with every variant the head dim has, on
the whole [B, H, N, d] problem), checked against the fp64 CPU oracle.

Sequence sweep: all 24 points (B*N = 16384 tokens, H = 16, N from 512 to 16384,
d in {64, 128}, both masks).  Head-dim sweep: all 12 points (B = 4, H = 16,
N = 4096, d in {64, 96, 128, 192, 256, 384}, both masks).

At each point, on sampled heads (the first, the last and one in the middle):
the forward on sampled rows (computed row by row by the oracle), and the
backward's dQ on sampled query rows and dK, dV on sampled key rows (the
row-restricted oracle, which needs no N x N matrix).  Every output element is
also checked to be finite.
"""

import numpy as np
import pytest

import oracle
from tiled_attention_tmem_gb300 import inputs as I

from helpers import GradCheck, check_fwd, head_f64, to_dev, to_f64

pytestmark = pytest.mark.gpu

POINTS = I.sweep_workloads() + I.head_dim_workloads()


def _variants(d):
    return (5, 7) if d in (64, 96, 128) else (7,)


@pytest.mark.parametrize("w", POINTS, ids=lambda w: w.name)
def test_sweep_point(w):
    import torch

    from tiled_attention_tmem_gb300 import api
    x = I.workload_inputs(w)
    q, k, v, do = (to_dev(t) for t in (x.q, x.k, x.v, x.do))
    o, lse = api.attention_forward(q, k, v, w.softmax_scale, w.causal)
    api.check_device_error()
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    rng = np.random.default_rng(w.seed)
    heads = sorted({(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 2)})
    edge = [0, 1, 127, 128, w.N - 1]
    refs = {}
    for b, h in heads:
        qf, kf, vf, dof = head_f64(x, b, h)
        rows = np.unique(np.concatenate([edge, rng.integers(0, w.N, size=27)]))
        o_ref, lse_ref = oracle.forward_rows(qf, kf, vf, w.softmax_scale, w.causal, 0, 0, rows)
        check_fwd(to_f64(o[b, h])[rows], to_f64(lse[b, h])[rows], o_ref, lse_ref, f"{w.name} b{b} h{h}")
        qrows = np.unique(np.concatenate([edge, rng.integers(0, w.N, size=11)]))
        krows = np.unique(np.concatenate([edge, rng.integers(0, w.N, size=11)]))
        refs[(b, h)] = (qrows, krows,
                        oracle.backward_rows(qf, kf, vf, dof, w.softmax_scale, w.causal, 0, 0, qrows, krows))
    for variant in _variants(w.d):
        dq, dk, dv = api.attention_backward(q, k, v, o, do, lse, w.softmax_scale, w.causal, variant=variant)
        api.check_device_error()
        for t in (dq, dk, dv):
            assert bool(torch.isfinite(t).all())
        chk = GradCheck(f"{w.name} v{variant}")
        for (b, h), (qrows, krows, ref) in refs.items():
            chk.add((to_f64(dq[b, h])[qrows], to_f64(dk[b, h])[krows], to_f64(dv[b, h])[krows]), ref)
        chk.check()
