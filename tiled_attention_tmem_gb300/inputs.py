"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds no attention arithmetic: it only draws i.i.d. normal numbers,
applies the workload's affine recipe (standard deviation, constant key shift)
and rounds them to bf16.  The same host bytes go to the GPU and, upcast exactly
to fp64, to the oracle.

Recipe (the pages give no inputs; this is the reading used everywhere):
  * generator: numpy ``Generator(PCG64(seed))``;
  * draw order: Q, K, V, dO, each ``standard_normal(shape, float32)`` of shape
    [B, H, N, d];
  * value = draw * sigma, plus ``k_shift`` on every element of K only;
  * rounded to bf16 with round-to-nearest-even.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    # bits + 0x7FFF + lsb, then >> 16: the largest non-NaN pattern (-inf, 0xFF800000)
    # stays below 2^32, so 32-bit arithmetic does not wrap; NaNs are set afterwards.
    rounded = (bits >> 16) & 1
    rounded += bits
    rounded += 0x7FFF
    rounded >>= 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


@dataclass(frozen=True)
class Workload:
    """One synthetic attention problem: shapes, mask, scale and the draw recipe."""

    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    sigma: float = 1.0
    k_shift: float = 0.0
    scale: float | None = None  # None means 1/sqrt(d)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d)

    @property
    def fwd_flops(self) -> float:
        """Nominal forward FLOPs 4*B*H*N^2*d, halved under the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def bwd_flops(self) -> float:
        """Nominal backward FLOPs: 2.5 times the forward, for either variant."""
        return 2.5 * self.fwd_flops


# The workloads attention is measured and checked on.
TINY = Workload("b1_h2_n256_d64", 1, 2, 256, 64, False, seed=1)
CAUSAL_2K = Workload("b4_h16_n2048_d128_causal", 4, 16, 2048, 128, True, seed=2)
KSHIFT_8K = Workload("b2_h16_n8192_d128_kshift3", 2, 16, 8192, 128, False, seed=3, k_shift=3.0)
HDIM256_4K = Workload("b2_h8_n4096_d256_causal_sigma0.5", 2, 8, 4096, 256, True,
                      seed=4, sigma=0.5, scale=1.0 / 16.0)
# One long head: fewer query blocks than SMs, the case the split-KV forward serves.
LONG_1H_16K = Workload("b1_h1_n16384_d128_causal", 1, 1, 16384, 128, True, seed=5)
LONG_1H_8K_D256 = Workload("b1_h1_n8192_d256_causal_sigma0.5", 1, 1, 8192, 256, True,
                           seed=6, sigma=0.5, scale=1.0 / 16.0)
# The largest head dim (lopsided tiles: 32 queries per dK/dV step, 32-key dQ tiles).
HDIM384_4K = Workload("b2_h8_n4096_d384_causal_sigma0.5", 2, 8, 4096, 384, True,
                      seed=7, sigma=0.5, scale=384 ** -0.5)


def sweep_workloads() -> list[Workload]:
    """Sequence sweep: B*N = 16384 tokens, H = 16, d in {64, 128}, both masks (24 points)."""
    out = []
    k = 0
    for d in (64, 128):
        for causal in (False, True):
            for n in (512, 1024, 2048, 4096, 8192, 16384):
                out.append(Workload(
                    f"sweep_n{n}_d{d}{'_causal' if causal else ''}",
                    16384 // n, 16, n, d, causal, seed=100 + k))
                k += 1
    return out


def head_dim_workloads() -> list[Workload]:
    """Head-dim sweep: B=4, H=16, N=4096, d in {64, 96, 128, 192, 256, 384}, both masks (12 points)."""
    out = []
    k = 0
    for d in (64, 96, 128, 192, 256, 384):
        for causal in (False, True):
            out.append(Workload(f"hdim_n4096_d{d}{'_causal' if causal else ''}", 4, 16, 4096, d, causal,
                                seed=200 + k))
            k += 1
    return out


WORKLOADS = {w.name: w for w in [TINY, CAUSAL_2K, KSHIFT_8K, HDIM256_4K, LONG_1H_16K, LONG_1H_8K_D256, HDIM384_4K]
             + sweep_workloads() + head_dim_workloads()}


@dataclass
class HostInputs:
    """bf16 bit patterns (uint16) of Q, K, V, dO, each [B, H, N, d] C-contiguous."""

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray
    extra: dict = field(default_factory=dict)

    def as_f64(self):
        return (bf16_bits_to_f64(self.q), bf16_bits_to_f64(self.k),
                bf16_bits_to_f64(self.v), bf16_bits_to_f64(self.do))


def make_inputs(B: int, H: int, N: int, d: int, seed: int,
                sigma: float = 1.0, k_shift: float = 0.0) -> HostInputs:
    """Draw Q, K, V, dO by the recipe in the module docstring."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (B, H, N, d)
    out = []
    for name in ("q", "k", "v", "do"):
        x = rng.standard_normal(shape, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        if name == "k" and k_shift != 0.0:
            x += np.float32(k_shift)
        out.append(f32_to_bf16_bits(x))
    return HostInputs(*out)


def workload_inputs(w: Workload) -> HostInputs:
    return make_inputs(w.B, w.H, w.N, w.d, w.seed, w.sigma, w.k_shift)
