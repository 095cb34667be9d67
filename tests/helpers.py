"""Shared test helpers: host<->device marshalling and tolerance checks."""

from __future__ import annotations

import numpy as np

from tiled_attention_tmem_gb300 import inputs as I

# Tolerances stated for this method: O max abs error <= 1e-2, LSE max abs error
# <= 1e-3, dQ/dK/dV max abs error <= 2e-2 * max|ref| (per tensor).
TOL_O = 1e-2
TOL_LSE = 1e-3
TOL_GRAD_REL = 2e-2


def to_dev(bits, device="cuda:0"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_f64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return I.bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.double().cpu().numpy()


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if not np.all(np.isfinite(a)):
        return float("inf")
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def check_fwd(o, lse, o_ref, lse_ref, what=""):
    eo = max_abs(o, o_ref)
    el = max_abs(lse, lse_ref)
    assert eo <= TOL_O, f"{what} O max abs err {eo:.3e} > {TOL_O}"
    assert el <= TOL_LSE, f"{what} LSE max abs err {el:.3e} > {TOL_LSE}"
    return eo, el


def check_grads(got, ref, what=""):
    # A tensor whose reference is identically zero (N = 1 gives dQ = dK = 0 exactly)
    # would be held to exactly zero by the relative bound; fp32 rounding of dP - D
    # leaves ~1e-6 there, so it is held to the largest gradient reference instead.
    scales = [float(np.max(np.abs(r))) if r.size else 0.0 for r in ref]
    floor = max(scales)
    out = []
    for name, g, r, s in zip(("dQ", "dK", "dV"), got, ref, scales):
        scale = s if s > 0 else floor
        e = max_abs(g, r)
        assert e <= TOL_GRAD_REL * scale, f"{what} {name} max abs err {e:.3e} > {TOL_GRAD_REL}*{scale:.3e}"
        out.append(e / scale if scale else 0.0)
    return out


def head_f64(x, b, h):
    """fp64 copies of Q, K, V, dO of head (b, h) only, shaped [1, 1, N, d] (for the oracle)."""
    return tuple(I.bf16_bits_to_f64(t[b:b + 1, h:h + 1]) for t in (x.q, x.k, x.v, x.do))


class GradCheck:
    """Collects (got, ref) pieces of dQ, dK, dV from several heads or rows and checks
    them at the end against one bound per tensor: max abs error <= 2e-2 * max|ref|,
    with max|ref| taken over everything collected for that tensor (the whole tensor
    when every element is checked; the sampled elements otherwise, which is stricter).
    """

    def __init__(self, what=""):
        self.what = what
        self.err = [0.0, 0.0, 0.0]
        self.scale = [0.0, 0.0, 0.0]

    def add(self, got, ref):
        for t, (g, r) in enumerate(zip(got, ref)):
            r = np.asarray(r, dtype=np.float64)
            if r.size == 0:
                continue
            self.err[t] = max(self.err[t], max_abs(g, r))
            self.scale[t] = max(self.scale[t], float(np.max(np.abs(r))))

    def check(self):
        floor = max(self.scale)
        for name, e, s in zip(("dQ", "dK", "dV"), self.err, self.scale):
            scale = s if s > 0 else floor
            assert e <= TOL_GRAD_REL * scale, f"{self.what} {name} max abs err {e:.3e} > {TOL_GRAD_REL}*{scale:.3e}"
        return [e / (s if s > 0 else floor) for e, s in zip(self.err, self.scale)]
