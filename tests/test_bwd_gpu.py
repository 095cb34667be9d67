"""Backward parity (5-GEMM and 7-GEMM) through the C ABI against the fp64 CPU oracle."""

import numpy as np
import pytest

import oracle
from tiled_attention_tmem_gb300 import inputs as I

from helpers import GradCheck, check_grads, head_f64, to_dev, to_f64

pytestmark = pytest.mark.gpu

V5, V7 = 5, 7

SMALL = [
    # (B, H, N, d, causal, sigma, k_shift, scale)
    (1, 2, 256, 64, False, 1.0, 0.0, None),
    (1, 2, 256, 64, True, 1.0, 0.0, None),
    (2, 3, 200, 64, True, 1.0, 0.0, None),
    (1, 2, 384, 128, True, 1.0, 0.0, None),
    (1, 2, 333, 128, False, 1.0, 0.0, None),
    (1, 1, 512, 128, False, 1.0, 3.0, None),
    (1, 1, 129, 128, True, 1.0, 0.0, None),
    (1, 1, 1, 64, False, 1.0, 0.0, None),
    (1, 1, 17, 128, True, 1.0, 0.0, None),
    (1, 2, 256, 256, True, 0.5, 0.0, 1.0 / 16),
    (1, 1, 300, 256, False, 1.0, 0.0, None),
    # head dims 96 (zero-padded 128 tiles) and 192 (its own 192-column tiles)
    (1, 2, 300, 96, True, 1.0, 0.0, None),
    (2, 1, 256, 96, False, 1.0, 3.0, None),
    (1, 2, 200, 192, True, 1.0, 0.0, None),
    (1, 1, 384, 192, False, 0.5, 0.0, None),
    (1, 2, 17, 192, True, 1.0, 0.0, None),
    (1, 1, 1, 256, False, 1.0, 0.0, None),
    (2, 1, 65, 256, True, 0.5, 0.0, 1.0 / 16),
    # head dim 384 (dV and dK in three column parts, dQ in two), both masks
    (1, 1, 1, 384, False, 1.0, 0.0, None),
    (1, 2, 1, 384, True, 1.0, 0.0, None),
    (1, 1, 129, 384, False, 1.0, 0.0, None),
    (1, 2, 129, 384, True, 1.0, 0.0, None),
    (1, 1, 1024, 384, False, 1.0, 0.0, None),
    (1, 1, 1024, 384, True, 1.0, 0.0, None),
    (2, 1, 333, 384, True, 0.5, 3.0, 1.0 / 20),
    # more work items than SMs: each persistent CTA claims several, short ones among them
    (2, 96, 256, 256, True, 0.5, 0.0, 1.0 / 16),
    (1, 160, 130, 384, True, 0.5, 0.0, None),
    (1, 200, 256, 128, True, 1.0, 0.0, None),
]


def _variants(d):
    return (V5, V7) if d in (64, 96, 128) else (V7,)


def _fwd_bwd(x, B, H, N, d, scale, causal, variant, o_lse=None):
    from tiled_attention_tmem_gb300 import api
    q, k, v, do = (to_dev(t) for t in (x.q, x.k, x.v, x.do))
    if o_lse is None:
        o, lse = api.attention_forward(q, k, v, scale, causal)
    else:
        o, lse = o_lse
    grads = api.attention_backward(q, k, v, o, do, lse, scale, causal, variant=variant)
    api.check_device_error()
    return grads


def _cases():
    for c in SMALL:
        for var in _variants(c[3]):
            yield c + (var,)


@pytest.mark.parametrize("case", list(_cases()),
                         ids=lambda c: "b{}h{}n{}d{}{}-v{}".format(*c[:4], "c" if c[4] else "", c[8]))
def test_backward_small_end_to_end(case):
    """The GPU backward consumes the GPU forward's O and LSE; the oracle uses its own."""
    B, H, N, d, causal, sigma, shift, scale, variant = case
    scale = scale if scale is not None else 1.0 / np.sqrt(d)
    x = I.make_inputs(B, H, N, d, seed=2000 + N + d, sigma=sigma, k_shift=shift)
    dq, dk, dv = _fwd_bwd(x, B, H, N, d, scale, causal, variant)
    qf, kf, vf, dof = x.as_f64()
    ref = oracle.backward(qf, kf, vf, dof, scale, causal)
    check_grads((to_f64(dq), to_f64(dk), to_f64(dv)), ref, f"{case}")


@pytest.mark.parametrize("variant", [V5, V7])
def test_backward_isolated_from_oracle_forward(variant):
    """The GPU backward fed bf16(O_ref) and fp32(LSE_ref) from the oracle."""
    import torch
    B, H, N, d, causal = 1, 2, 320, 128, True
    scale = 1.0 / np.sqrt(d)
    x = I.make_inputs(B, H, N, d, seed=77)
    qf, kf, vf, dof = x.as_f64()
    o_ref, lse_ref = oracle.forward(qf, kf, vf, scale, causal)
    o_dev = to_dev(I.f32_to_bf16_bits(o_ref.astype(np.float32)))
    lse_dev = torch.from_numpy(lse_ref.astype(np.float32)).cuda()
    dq, dk, dv = _fwd_bwd(x, B, H, N, d, scale, causal, variant, o_lse=(o_dev, lse_dev))
    ref = oracle.backward(qf, kf, vf, dof, scale, causal)
    check_grads((to_f64(dq), to_f64(dk), to_f64(dv)), ref, "isolated")


def test_seven_gemm_is_bitwise_reproducible():
    x = I.make_inputs(2, 2, 640, 128, seed=9)
    a = _fwd_bwd(x, 2, 2, 640, 128, 0.0884, True, V7)
    b = _fwd_bwd(x, 2, 2, 640, 128, 0.0884, True, V7)
    for u, w in zip(a, b):
        assert np.array_equal(to_f64(u), to_f64(w))


def test_seven_gemm_is_bitwise_reproducible_at_d384():
    x = I.make_inputs(1, 2, 700, 384, seed=19)
    a = _fwd_bwd(x, 1, 2, 700, 384, 384 ** -0.5, True, V7)
    b = _fwd_bwd(x, 1, 2, 700, 384, 384 ** -0.5, True, V7)
    for u, w in zip(a, b):
        assert np.array_equal(to_f64(u), to_f64(w))


def test_five_and_seven_agree():
    x = I.make_inputs(1, 4, 512, 64, seed=10)
    a = _fwd_bwd(x, 1, 4, 512, 64, 0.125, False, V5)
    b = _fwd_bwd(x, 1, 4, 512, 64, 0.125, False, V7)
    for u, w in zip(a, b):
        u64, w64 = to_f64(u), to_f64(w)
        assert np.max(np.abs(u64 - w64)) <= 1e-2 * np.max(np.abs(w64))


# Full-size workloads in the bench's launch configuration (fa_fwd then fa_bwd on the
# whole [B, H, N, d] problem), every variant the head dim has.  Every head is checked
# against the oracle: element by element where its N x N matrices fit (the N = 2048
# and the d = 256 workloads), and on sampled query rows (dQ) and key rows (dK, dV)
# computed by the row-restricted oracle for the N = 8192 workload.
FULL_EVERY_ROW = [I.CAUSAL_2K, I.HDIM256_4K]


@pytest.mark.parametrize("w", FULL_EVERY_ROW, ids=lambda w: w.name)
def test_backward_full_size_every_head_every_row(w):
    x = I.workload_inputs(w)
    refs = {}
    for b in range(w.B):
        for h in range(w.H):
            qf, kf, vf, dof = head_f64(x, b, h)
            parts = oracle.backward_parts(qf[0, 0], kf[0, 0], vf[0, 0], dof[0, 0], w.softmax_scale, w.causal)
            refs[(b, h)] = (parts["dQ"], parts["dK"], parts["dV"])
            del parts
    for variant in _variants(w.d):
        dq, dk, dv = _fwd_bwd(x, w.B, w.H, w.N, w.d, w.softmax_scale, w.causal, variant)
        g = [to_f64(t) for t in (dq, dk, dv)]
        chk = GradCheck(f"{w.name} v{variant}")
        for (b, h), ref in refs.items():
            chk.add([t[b, h] for t in g], ref)
        chk.check()


def test_backward_full_size_every_head_sampled_rows():
    """B=2, H=16, N=8192 with keys shifted by +3: every head, sampled rows, both variants."""
    w = I.KSHIFT_8K
    x = I.workload_inputs(w)
    rng = np.random.default_rng(w.seed)
    refs = {}
    for b in range(w.B):
        for h in range(w.H):
            edge = [0, 127, 128, w.N - 1]
            qrows = np.unique(np.concatenate([edge, rng.integers(0, w.N, size=20)]))
            krows = np.unique(np.concatenate([edge, rng.integers(0, w.N, size=20)]))
            qf, kf, vf, dof = head_f64(x, b, h)
            refs[(b, h)] = (qrows, krows,
                            oracle.backward_rows(qf, kf, vf, dof, w.softmax_scale, w.causal, 0, 0, qrows, krows))
    for variant in _variants(w.d):
        dq, dk, dv = _fwd_bwd(x, w.B, w.H, w.N, w.d, w.softmax_scale, w.causal, variant)
        g = [to_f64(t) for t in (dq, dk, dv)]
        for t in g:
            assert np.all(np.isfinite(t))
        chk = GradCheck(f"{w.name} v{variant}")
        for (b, h), (qrows, krows, ref) in refs.items():
            chk.add((g[0][b, h, qrows], g[1][b, h, krows], g[2][b, h, krows]), ref)
        chk.check()
