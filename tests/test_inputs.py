"""The seeded input generator: determinism, recipe, and bf16 rounding."""

import numpy as np
import pytest

from tiled_attention_tmem_gb300 import inputs as I


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 10,
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38, -1e-40, 65504.0], np.float32),
    ])
    ours = I.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = I.bf16_bits_to_f32(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_ties_round_to_even():
    # 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7: rounds to 1 (even).
    assert I.f32_to_bf16_bits(np.float32(1.0 + 2**-8)) == 0x3F80
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: rounds up to the even one.
    assert I.f32_to_bf16_bits(np.float32(1.0 + 3 * 2**-8)) == 0x3F82


def test_deterministic_and_recipe():
    a = I.make_inputs(1, 2, 16, 8, seed=5, sigma=0.5, k_shift=3.0)
    b = I.make_inputs(1, 2, 16, 8, seed=5, sigma=0.5, k_shift=3.0)
    for x, y in zip((a.q, a.k, a.v, a.do), (b.q, b.k, b.v, b.do)):
        np.testing.assert_array_equal(x, y)
    q, k, v, do = a.as_f64()
    assert abs(k.mean() - 3.0) < 0.3
    assert abs(q.std() - 0.5) < 0.15
    c = I.make_inputs(1, 2, 16, 8, seed=6)
    assert not np.array_equal(a.q, c.q)


def test_workload_table():
    sweep = I.sweep_workloads()
    assert len(sweep) == 24
    assert all(w.B * w.N == 16384 and w.H == 16 for w in sweep)
    w = I.WORKLOADS["b4_h16_n2048_d128_causal"]
    assert w.fwd_flops == 4 * 4 * 16 * 2048 ** 2 * 128 / 2
    assert w.bwd_flops == 2.5 * w.fwd_flops
    assert I.HDIM256_4K.softmax_scale == 1 / 16
