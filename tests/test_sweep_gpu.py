"""Parity on the sequence-sweep configuration: B*N = 16384 tokens, H = 16,
d in {64, 128}, both masks, N from 512 to 16384 (the shapes and launch
configuration the sweep measures), checked against the fp64 CPU oracle.

At each point: the forward on sampled rows of three heads (the oracle computes
them row by row), and, wherever the oracle's materialised N x N matrices stay
small (N <= 2048), the backward on whole sampled heads for every variant.
"""

import numpy as np
import pytest

import oracle
from tiled_attention_tmem_gb300 import inputs as I

from helpers import check_fwd, check_grads, to_dev, to_f64

pytestmark = pytest.mark.gpu

SWEEP = {w.name: w for w in I.sweep_workloads()}
POINTS = ["sweep_n512_d64_causal", "sweep_n512_d128", "sweep_n2048_d64",
          "sweep_n16384_d64", "sweep_n16384_d128_causal"]


@pytest.mark.parametrize("name", POINTS)
def test_sweep_point(name):
    from tiled_attention_tmem_gb300 import api
    w = SWEEP[name]
    x = I.workload_inputs(w)
    qf, kf, vf, dof = x.as_f64()
    q, k, v, do = (to_dev(t) for t in (x.q, x.k, x.v, x.do))
    o, lse = api.attention_forward(q, k, v, w.softmax_scale, w.causal)
    api.check_device_error()
    o64, l64 = to_f64(o), to_f64(lse)
    assert np.all(np.isfinite(o64)) and np.all(np.isfinite(l64))
    rng = np.random.default_rng(w.seed)
    for b, h in [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 2)]:
        rows = np.unique(np.concatenate([[0, 1, 127, 128, w.N - 1], rng.integers(0, w.N, size=27)]))
        o_ref, lse_ref = oracle.forward_rows(qf, kf, vf, w.softmax_scale, w.causal, b, h, rows)
        check_fwd(o64[b, h, rows], l64[b, h, rows], o_ref, lse_ref, f"{name} b{b} h{h}")
    if w.N > 2048:
        return
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    refs = {}
    for b, h in heads:
        parts = oracle.backward_parts(qf[b, h], kf[b, h], vf[b, h], dof[b, h], w.softmax_scale, w.causal)
        refs[(b, h)] = (parts["dQ"], parts["dK"], parts["dV"])
    for variant in (5, 7):
        dq, dk, dv = api.attention_backward(q, k, v, o, do, lse, w.softmax_scale, w.causal, variant=variant)
        api.check_device_error()
        g = [to_f64(t) for t in (dq, dk, dv)]
        for b, h in heads:
            check_grads([t[b, h] for t in g], refs[(b, h)], f"{name} v{variant} b{b} h{h}")
        for t in g:
            assert np.all(np.isfinite(t))
