"""Query-range split of the dK/dV kernel and key-range split of the 7-GEMM dQ
kernel (few heads, long sequences) against the fp64 CPU oracle, through the C ABI.

With fewer key tiles than SMs the library cuts each key tile's query tiles into
parts, runs each part as its own work item writing fp32 partial dK and dV, and
adds the parts in a separate kernel; the dQ kernel likewise cuts each query
tile's key tiles into parts with fp32 partial dQ.  These shapes are ones where
the library's rules split (checked through the launch count: one extra kernel
per split)."""

import numpy as np
import pytest

import oracle
from tiled_attention_tmem_gb300 import binding as b
from tiled_attention_tmem_gb300 import inputs as I

from helpers import GradCheck, check_grads, head_f64, to_dev, to_f64

pytestmark = pytest.mark.gpu

# (B, H, N, d, causal, variant)
CASES = [
    (1, 1, 4096, 128, True, 5),
    (1, 1, 4096, 128, True, 7),
    (1, 1, 3000, 96, True, 5),
    (1, 1, 2500, 64, True, 5),
    (1, 1, 4096, 64, True, 7),
    (1, 1, 4096, 256, True, 7),
    (1, 1, 3333, 192, True, 7),
    (1, 1, 2048, 384, True, 7),
]


def _split_used(B, H, N, d, causal, variant):
    parts = b.fa_bwd_query_parts(B, H, N, d, int(causal), variant)
    kparts = b.fa_bwd_key_parts(B, H, N, d, int(causal), variant)
    return parts > 1 and b.fa_bwd_launches(B, H, N, d, variant, int(causal)) == 4 + (kparts > 1)


def _key_split_used(B, H, N, d, causal):
    kparts = b.fa_bwd_key_parts(B, H, N, d, int(causal), 7)
    qparts = b.fa_bwd_query_parts(B, H, N, d, int(causal), 7)
    return kparts > 1 and b.fa_bwd_launches(B, H, N, d, 7, int(causal)) == 4 + (qparts > 1)


def _run(x, B, H, N, d, causal, variant):
    from tiled_attention_tmem_gb300 import api
    q, k, v, do = (to_dev(t) for t in (x.q, x.k, x.v, x.do))
    scale = 1.0 / np.sqrt(d)
    o, lse = api.attention_forward(q, k, v, scale, causal)
    grads = api.attention_backward(q, k, v, o, do, lse, scale, causal, variant=variant)
    api.check_device_error()
    return [to_f64(t) for t in grads]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}n{}d{}{}-v{}".format(*c[:4], "c" if c[4] else "", c[5]))
def test_split_backward_matches_oracle(case):
    B, H, N, d, causal, variant = case
    assert _split_used(B, H, N, d, causal, variant), "the cost model no longer splits this shape"
    x = I.make_inputs(B, H, N, d, seed=3100 + N + d)
    got = _run(x, B, H, N, d, causal, variant)
    qf, kf, vf, dof = head_f64(x, 0, 0)
    parts = oracle.backward_parts(qf[0, 0], kf[0, 0], vf[0, 0], dof[0, 0], 1.0 / np.sqrt(d), causal)
    check_grads([t[0, 0] for t in got], (parts["dQ"], parts["dK"], parts["dV"]), f"{case}")


def test_split_seven_gemm_is_bitwise_reproducible():
    B, H, N, d, causal = 1, 1, 4096, 128, True
    assert _split_used(B, H, N, d, causal, 7)
    x = I.make_inputs(B, H, N, d, seed=3200)
    a = _run(x, B, H, N, d, causal, 7)
    c = _run(x, B, H, N, d, causal, 7)
    for u, w in zip(a, c):
        assert np.array_equal(u, w)


def test_split_long_single_head_sampled_rows():
    """One head of 16384 rows under the causal mask (the few-heads workload), both
    variants, on sampled rows of the row-restricted oracle."""
    w = I.LONG_1H_16K
    x = I.workload_inputs(w)
    rng = np.random.default_rng(w.seed)
    edge = [0, 127, 128, w.N - 1]
    qrows = np.unique(np.concatenate([edge, rng.integers(0, w.N, size=40)]))
    krows = np.unique(np.concatenate([edge, rng.integers(0, w.N, size=40)]))
    qf, kf, vf, dof = head_f64(x, 0, 0)
    ref = oracle.backward_rows(qf, kf, vf, dof, w.softmax_scale, w.causal, 0, 0, qrows, krows)
    for variant in (5, 7):
        assert _split_used(w.B, w.H, w.N, w.d, w.causal, variant)
        g = _run(x, w.B, w.H, w.N, w.d, w.causal, variant)
        chk = GradCheck(f"{w.name} v{variant}")
        chk.add((g[0][0, 0, qrows], g[1][0, 0, krows], g[2][0, 0, krows]), ref)
        chk.check()


@pytest.mark.parametrize("parts", [2, 5, 8, 16])
def test_forced_part_counts_match_oracle(parts):
    """Every part count through the benchmark hook, including more parts than some
    key tiles have query tiles (empty parts write zero partial sums)."""
    B, H, N, d, causal = 1, 2, 1100, 128, True
    x = I.make_inputs(B, H, N, d, seed=3300 + parts)
    assert b.fa_bwd_force_query_parts(parts) == b.FA_OK
    try:
        assert b.fa_bwd_query_parts(B, H, N, d, 1, 5) == parts
        got5 = _run(x, B, H, N, d, causal, 5)
        got7 = _run(x, B, H, N, d, causal, 7)
    finally:
        b.fa_bwd_force_query_parts(0)
    qf, kf, vf, dof = x.as_f64()
    ref = oracle.backward(qf, kf, vf, dof, 1.0 / np.sqrt(d), causal)
    check_grads(got5, ref, f"parts {parts} v5")
    check_grads(got7, ref, f"parts {parts} v7")


# (B, H, N, d, causal): the 7-GEMM dQ kernel's key split at every dQ configuration
# (d = 64 and 128 with S and dP from shared-memory dO, 192 and 256 with dO in
# TMEM, 384 with two dQ column parts), both masks and ragged lengths.
KEY_CASES = [
    (1, 1, 4096, 256, True),
    (1, 2, 2500, 192, True),
    (1, 1, 3000, 384, True),
    (1, 1, 2048, 64, True),
    (1, 1, 1800, 96, True),
    (1, 1, 4096, 256, False),
    (1, 1, 2200, 128, False),
]


@pytest.mark.parametrize("case", KEY_CASES, ids=lambda c: "b{}h{}n{}d{}{}".format(*c[:4], "c" if c[4] else ""))
def test_key_split_backward_matches_oracle(case):
    B, H, N, d, causal = case
    assert _key_split_used(B, H, N, d, causal), "the rule no longer splits this shape's keys"
    x = I.make_inputs(B, H, N, d, seed=3400 + N + d)
    got = _run(x, B, H, N, d, causal, 7)
    chk = GradCheck(f"{case}")
    for h in range(H):
        qf, kf, vf, dof = head_f64(x, 0, h)
        parts = oracle.backward_parts(qf[0, 0], kf[0, 0], vf[0, 0], dof[0, 0], 1.0 / np.sqrt(d), causal)
        chk.add([t[0, h] for t in got], (parts["dQ"], parts["dK"], parts["dV"]))
    chk.check()


@pytest.mark.parametrize("d", [128, 256, 384])
@pytest.mark.parametrize("parts", [2, 5, 16])
def test_forced_key_part_counts_match_oracle(parts, d):
    """Key-part counts through the benchmark hook, including more parts than the
    first query tiles have key tiles (empty parts write zero partial sums); the
    query split stays off so that only the dQ kernel is split."""
    B, H, N, causal = 1, 2, 1100, True
    x = I.make_inputs(B, H, N, d, seed=3500 + parts + d)
    assert b.fa_bwd_force_key_parts(parts) == b.FA_OK
    assert b.fa_bwd_force_query_parts(1) == b.FA_OK
    try:
        assert b.fa_bwd_key_parts(B, H, N, d, 1, 7) == parts
        assert b.fa_bwd_launches(B, H, N, d, 7, 1) == 4
        got = _run(x, B, H, N, d, causal, 7)
    finally:
        b.fa_bwd_force_key_parts(0)
        b.fa_bwd_force_query_parts(0)
    qf, kf, vf, dof = x.as_f64()
    ref = oracle.backward(qf, kf, vf, dof, 1.0 / np.sqrt(d), causal)
    check_grads(got, ref, f"key parts {parts} d{d}")


def test_key_split_is_bitwise_reproducible_and_only_changes_dq():
    """The key split sums its parts in a fixed order: two runs agree bit for bit, and
    dK, dV (from the dK/dV kernel, whose split is held fixed) are bit-equal to the
    run without a key split."""
    B, H, N, d, causal = 1, 1, 4096, 256, True
    x = I.make_inputs(B, H, N, d, seed=3600)
    assert b.fa_bwd_force_query_parts(2) == b.FA_OK
    try:
        assert b.fa_bwd_force_key_parts(1) == b.FA_OK
        plain = _run(x, B, H, N, d, causal, 7)
        assert b.fa_bwd_force_key_parts(6) == b.FA_OK
        a = _run(x, B, H, N, d, causal, 7)
        c = _run(x, B, H, N, d, causal, 7)
    finally:
        b.fa_bwd_force_key_parts(0)
        b.fa_bwd_force_query_parts(0)
    for u, w in zip(a, c):
        assert np.array_equal(u, w)
    assert np.array_equal(a[1], plain[1]) and np.array_equal(a[2], plain[2])
    scale = np.abs(plain[0]).max()
    assert np.abs(a[0] - plain[0]).max() <= 2e-2 * scale
