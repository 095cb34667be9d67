"""Pins for the CPU oracle: closed forms, invariants, brute force and finite differences.

Each check ties the oracle to something other than itself, chosen so that a
plausible mistake (a dropped scale, a wrong sign, an off-by-one in the causal
mask, a transposed operand, a missing max in LSE) fails at least one of them.
``test_planted_mistakes_are_caught`` plants such mistakes in copies of the
oracle's formulas and checks that the pins notice.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import attention as A

RNG = np.random.default_rng(12345)


def rand(*shape, scale=1.0, rng=None):
    r = rng if rng is not None else RNG
    return r.standard_normal(shape) * scale


# ---------------------------------------------------------------- (1) blockwise merge


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,blocks", [
    (64, [1] * 64), (63, [3] * 21), (70, [7] * 10), (64, [16] * 4), (64, [64]),
    (64, [5, 20, 1, 30, 8]), (33, [1, 31, 1]),
])
def test_online_merge_equals_direct(causal, n, blocks):
    """ELI5 article: merging per-block m and l gives exactly the direct softmax."""
    d = 8
    q, k, v = rand(n, d), rand(n, d), rand(n, d)
    o_ref, lse_ref = A.forward(q[None, None], k[None, None], v[None, None], 0.3, causal)
    o, lse = oracle.blockwise_forward(q, k, v, 0.3, causal, blocks)
    np.testing.assert_allclose(o, o_ref[0, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref[0, 0], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_online_merge_with_large_max_jumps(causal):
    """Scores whose row maximum jumps by more than 20 between blocks."""
    n, d = 48, 4
    q = rand(n, d)
    k = rand(n, d)
    # Later key blocks have much larger scores for every query.
    for blk in range(6):
        k[blk * 8:(blk + 1) * 8] += 25.0 * blk * np.sign(q.mean(0))[None, :] / d
    q = np.abs(q) + 0.5
    k = np.abs(k)
    k[8:] *= 4.0
    v = rand(n, d)
    s = A.scores(q[None, None], k[None, None], 1.0, False)[0, 0]
    blockmax = [s[:, i * 8:(i + 1) * 8].max(1) for i in range(6)]
    assert np.max(blockmax[5] - blockmax[0]) > 20.0
    o_ref, lse_ref = A.forward(q[None, None], k[None, None], v[None, None], 1.0, causal)
    for blocks in ([8] * 6, [1] * 48, [16, 32]):
        o, lse = oracle.blockwise_forward(q, k, v, 1.0, causal, blocks)
        np.testing.assert_allclose(o, o_ref[0, 0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref[0, 0], rtol=1e-12)


def test_random_partitions_merge():
    rng = np.random.default_rng(7)
    for trial in range(20):
        n = int(rng.integers(1, 90))
        cuts = sorted(set(rng.integers(1, n, size=int(rng.integers(0, 6))).tolist())) if n > 1 else []
        edges = [0] + cuts + [n]
        blocks = [b - a for a, b in zip(edges[:-1], edges[1:])]
        q, k, v = rand(n, 5, rng=rng), rand(n, 5, rng=rng), rand(n, 5, rng=rng)
        causal = bool(trial % 2)
        o_ref, lse_ref = A.forward(q[None, None], k[None, None], v[None, None], 0.7, causal)
        o, lse = oracle.blockwise_forward(q, k, v, 0.7, causal, blocks)
        np.testing.assert_allclose(o, o_ref[0, 0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref[0, 0], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,parts", [
    (64, [32, 32]), (64, [16] * 4), (70, [7] * 10), (64, [64]), (65, [0, 30, 0, 35, 0]),
    (200, [128, 72]), (33, [1, 31, 1]), (256, [64] * 4), (5, [1] * 5),
])
def test_split_forward_equals_direct(causal, n, parts):
    """Key ranges finished on their own and merged by their log-sum-exps give the
    direct softmax; under the causal mask later ranges are fully masked for the
    early rows (L_s = -inf, weight 0), and empty ranges contribute nothing."""
    d = 8
    q, k, v = rand(n, d), rand(n, d), rand(n, d)
    o_ref, lse_ref = A.forward(q[None, None], k[None, None], v[None, None], 0.3, causal)
    o, lse = oracle.split_forward(q, k, v, 0.3, causal, parts)
    np.testing.assert_allclose(o, o_ref[0, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref[0, 0], rtol=1e-12, atol=1e-13)
    o_b, lse_b = oracle.blockwise_forward(q, k, v, 0.3, causal, [p for p in parts if p])
    np.testing.assert_allclose(o, o_b, rtol=1e-12, atol=1e-13)


def test_split_forward_far_apart_maxima_and_random_parts():
    """Part maxima more than 30 apart (keys shifted along q), and random partitions."""
    rng = np.random.default_rng(21)
    n, d = 96, 4
    q = np.abs(rand(n, d, rng=rng)) + 0.5
    k = rand(n, d, rng=rng)
    k[48:] += 20.0  # the second half of the keys scores far higher for every query
    v = rand(n, d, rng=rng)
    s = A.scores(q[None, None], k[None, None], 1.0, False)[0, 0]
    assert np.min(s[:, 48:].max(1) - s[:, :48].max(1)) > 30.0
    for causal in (False, True):
        o_ref, lse_ref = A.forward(q[None, None], k[None, None], v[None, None], 1.0, causal)
        for parts in ([48, 48], [8] * 12, [95, 1], [1, 95]):
            o, lse = oracle.split_forward(q, k, v, 1.0, causal, parts)
            np.testing.assert_allclose(o, o_ref[0, 0], rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(lse, lse_ref[0, 0], rtol=1e-12)
    for trial in range(12):
        n = int(rng.integers(2, 80))
        cuts = sorted(rng.integers(0, n + 1, size=int(rng.integers(1, 7))).tolist())
        edges = [0] + cuts + [n]
        parts = [b - a for a, b in zip(edges[:-1], edges[1:])]
        q, k, v = rand(n, 3, rng=rng), rand(n, 3, rng=rng), rand(n, 3, rng=rng)
        causal = bool(trial % 2)
        o_ref, lse_ref = A.forward(q[None, None], k[None, None], v[None, None], 0.9, causal)
        o, lse = oracle.split_forward(q, k, v, 0.9, causal, parts)
        np.testing.assert_allclose(o, o_ref[0, 0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref[0, 0], rtol=1e-12, atol=1e-13)


def test_split_merge_mistakes_are_caught():
    """Plausible mistakes in the part merge fail the equality with the direct
    definition: weights not renormalised by their sum, part LSEs in log2 mixed
    with natural exponentials, and a fully masked part given weight exp(0)."""
    n, d = 64, 6
    q, k, v = rand(n, d), rand(n, d), rand(n, d)
    o_ref, lse_ref = A.forward(q[None, None], k[None, None], v[None, None], 0.4, True)
    parts = [(0, 32), (32, 64)]
    rows = np.arange(n)[:, None]
    o_s, l_s = [], []
    for a, b in parts:
        s = 0.4 * q @ k[a:b].T
        s = np.where(np.arange(a, b)[None, :] <= rows, s, -np.inf)
        m = s.max(1)
        seen = ~np.isneginf(m)
        p = np.exp(s - np.where(seen, m, 0.0)[:, None])
        l = p.sum(1)
        o = np.zeros((n, d))
        o[seen] = (p @ v[a:b])[seen] / l[seen][:, None]
        o_s.append(o)
        l_s.append(np.where(seen, np.where(seen, m, 0.0) + np.log(np.where(seen, l, 1.0)), -np.inf))
    L = np.stack(l_s)
    top = L.max(0)

    def merged(w):
        return np.einsum("sr,srd->rd", w, np.stack(o_s))

    w_ok = np.where(np.isneginf(L), 0.0, np.exp(L - top))
    good = merged(w_ok / w_ok.sum(0))
    np.testing.assert_allclose(good, o_ref[0, 0], rtol=1e-12, atol=1e-13)
    not_renormalised = merged(w_ok)
    assert np.max(np.abs(not_renormalised - o_ref[0, 0])) > 1e-3
    w_log2 = np.where(np.isneginf(L), 0.0, np.exp((L - top) / math.log(2.0)))
    log2_mixup = merged(w_log2 / w_log2.sum(0))
    assert np.max(np.abs(log2_mixup - o_ref[0, 0])) > 1e-3
    w_masked_one = np.where(np.isneginf(L), 1.0, np.exp(L - top))
    masked_weighted = merged(w_masked_one / w_masked_one.sum(0))
    assert np.max(np.abs(masked_weighted - o_ref[0, 0])) > 1e-3


def test_merge_partials_split_kv():
    """Two halves of the keys merged with the m/l algebra equal the whole."""
    n, d = 40, 6
    q, k, v = rand(n, d), rand(n, d), rand(n, d)
    o_ref, lse_ref = A.forward(q[None, None], k[None, None], v[None, None], 0.5, False)
    parts = []
    for sl in (slice(0, 17), slice(17, n)):
        s = 0.5 * q @ k[sl].T
        m = s.max(1)
        p = np.exp(s - m[:, None])
        parts.append((m, p.sum(1), p @ v[sl]))
    m, l, o = oracle.merge_partials(*parts[0], *parts[1])
    np.testing.assert_allclose(o / l[:, None], o_ref[0, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(m + np.log(l), lse_ref[0, 0], rtol=1e-12)


# ------------------------------------------------------- (2) rows of P and (3) D identity


@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    q, k = rand(2, 3, 37, 16), rand(2, 3, 37, 16)
    p = A.probabilities(q, k, 0.25, causal)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert np.all(p >= 0)
    if causal:
        assert np.all(p[..., np.triu_indices(37, 1)[0], np.triu_indices(37, 1)[1]] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_d_equals_rowsum_p_dp(causal):
    """D_i = sum_c dO_ic O_ic equals sum_j P_ij dP_ij (both are dO_i . sum_j P_ij V_j)."""
    n, d = 29, 12
    parts = A.backward_parts(rand(n, d), rand(n, d), rand(n, d), rand(n, d), 0.4, causal)
    lhs = parts["D"]
    rhs = np.sum(parts["P"] * parts["dP"], axis=1)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------ (4) finite differences


def _objective(q, k, v, do, scale, causal):
    o, _ = A.forward(q, k, v, scale, causal)
    return float(np.sum(o * do))


def _fd_errors(q, k, v, do, scale, causal, backward=A.backward):
    """Max |fd - analytic| / max|analytic| per tensor for f = sum(O * dO)."""
    grads = backward(q, k, v, do, scale, causal)
    errs = []
    for which, g in zip(range(3), grads):
        base = [q, k, v]
        fd = np.zeros_like(base[which])
        it = np.nditer(base[which], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x = base[which][idx]
            h = 1e-5 * max(1.0, abs(x))
            plus = [t.copy() for t in base]
            minus = [t.copy() for t in base]
            plus[which][idx] = x + h
            minus[which][idx] = x - h
            fd[idx] = (_objective(*plus, do, scale, causal) - _objective(*minus, do, scale, causal)) / (2 * h)
        # Below ~1e-9 central differences only see their own rounding noise
        # (machine epsilon * |f| / h); exactly-zero gradients (N = 1) are pinned
        # by the closed-form test instead.
        denom = max(np.max(np.abs(g)), 1e-9)
        errs.append(np.max(np.abs(fd - g)) / denom)
    return errs


@pytest.mark.parametrize("n", [1, 2, 5, 16])
@pytest.mark.parametrize("d", [1, 3, 8])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("scale_kind", ["rsqrt", "0.37"])
def test_finite_differences(n, d, causal, scale_kind):
    scale = 1.0 / math.sqrt(d) if scale_kind == "rsqrt" else 0.37
    rng = np.random.default_rng(n * 100 + d * 10 + int(causal))
    q, k, v, do = (rand(1, 1, n, d, rng=rng) for _ in range(4))
    errs = _fd_errors(q, k, v, do, scale, causal)
    for name, e in zip("QKV", errs):
        assert e <= 1e-6, f"d{name}: {e}"


# --------------------------------------------------------- (5) closed forms, invariants


def test_single_key():
    """N = 1: O = V, LSE = scale q.k, dQ = dK = 0, dV = dO."""
    q, k, v, do = (rand(2, 2, 1, 7) for _ in range(4))
    for causal in (False, True):
        o, lse = A.forward(q, k, v, 0.3, causal)
        np.testing.assert_allclose(o, v, rtol=1e-15)
        np.testing.assert_allclose(lse, 0.3 * np.sum(q * k, -1), rtol=1e-14)
        dq, dk, dv = A.backward(q, k, v, do, 0.3, causal)
        np.testing.assert_allclose(dq, 0, atol=1e-15)
        np.testing.assert_allclose(dk, 0, atol=1e-15)
        np.testing.assert_allclose(dv, do, rtol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_attention(causal):
    """Equal key rows (or scale 0): P is uniform over the visible keys."""
    n, d = 11, 5
    q, v = rand(1, 1, n, d), rand(1, 1, n, d)
    krow = rand(d)
    k = np.broadcast_to(krow, (1, 1, n, d)).copy()
    counts = np.arange(1, n + 1) if causal else np.full(n, n)
    cum = np.cumsum(v[0, 0], axis=0) if causal else np.broadcast_to(v[0, 0].sum(0), (n, d))
    mean_v = cum / counts[:, None]
    o, lse = A.forward(q, k, v, 0.6, causal)
    np.testing.assert_allclose(o[0, 0], mean_v, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], 0.6 * q[0, 0] @ krow + np.log(counts), rtol=1e-12)
    k2 = rand(1, 1, n, d)
    o0, lse0 = A.forward(q, k2, v, 0.0, causal)
    np.testing.assert_allclose(o0[0, 0], mean_v, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse0[0, 0], np.log(counts), rtol=1e-12)


def test_causal_first_row():
    q, k, v = rand(1, 2, 9, 4), rand(1, 2, 9, 4), rand(1, 2, 9, 4)
    o, lse = A.forward(q, k, v, 0.9, True)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], 0.9 * np.sum(q[:, :, 0] * k[:, :, 0], -1), rtol=1e-15)


def test_two_keys_closed_form():
    """N = 2, d = 1, no mask: softmax of two scores is a logistic function."""
    a, b = 0.8, -1.3
    q = np.array([a, b]).reshape(1, 1, 2, 1)
    k = np.array([0.5, 2.0]).reshape(1, 1, 2, 1)
    v = np.array([3.0, -1.0]).reshape(1, 1, 2, 1)
    scale = 0.75
    o, lse = A.forward(q, k, v, scale, False)
    for i, qi in enumerate((a, b)):
        s0, s1 = scale * qi * 0.5, scale * qi * 2.0
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        assert abs(o[0, 0, i, 0] - (3.0 * (1 - w1) - 1.0 * w1)) < 1e-14
        assert abs(lse[0, 0, i] - math.log(math.exp(s0) + math.exp(s1))) < 1e-14
    # Causal: row 0 sees only key 0.
    oc, _ = A.forward(q, k, v, scale, True)
    assert oc[0, 0, 0, 0] == 3.0


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    """K_j -> K_j + c leaves O, P and all gradients unchanged; LSE shifts by scale q.c."""
    n, d = 17, 6
    q, k, v, do = (rand(1, 1, n, d) for _ in range(4))
    c = rand(d) * 3.0
    o1, lse1 = A.forward(q, k, v, 0.5, causal)
    o2, lse2 = A.forward(q, k + c, v, 0.5, causal)
    np.testing.assert_allclose(o2, o1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse2, lse1 + 0.5 * (q @ c), rtol=1e-12, atol=1e-12)
    g1 = A.backward(q, k, v, do, 0.5, causal)
    g2 = A.backward(q, k + c, v, do, 0.5, causal)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(b, a, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sums_vanish(causal):
    """sum_j dS_ij = 0 for every row, hence sum_j dK_j = 0 per head."""
    n, d = 23, 9
    parts = A.backward_parts(rand(n, d), rand(n, d), rand(n, d), rand(n, d), 0.33, causal)
    np.testing.assert_allclose(parts["dS"].sum(1), 0, atol=1e-13)
    np.testing.assert_allclose(parts["dK"].sum(0), 0, atol=1e-12)


def test_affine_values():
    """V -> a V + 1 b^T gives O -> a O + b (rows of P sum to one)."""
    q, k, v = rand(1, 2, 13, 4), rand(1, 2, 13, 4), rand(1, 2, 13, 4)
    bvec = rand(4)
    for causal in (False, True):
        o, _ = A.forward(q, k, v, 0.8, causal)
        o2, _ = A.forward(q, k, -2.5 * v + bvec, 0.8, causal)
        np.testing.assert_allclose(o2, -2.5 * o + bvec, rtol=1e-12, atol=1e-12)


def test_permutation_equivariance():
    """Without a mask, permuting keys and values together changes nothing but the
    order of dK and dV; permuting queries (with dO) permutes O, LSE and dQ alike."""
    n, d = 19, 7
    q, k, v, do = (rand(1, 1, n, d) for _ in range(4))
    perm = np.random.default_rng(7).permutation(n)
    o, lse = A.forward(q, k, v, 0.4, False)
    dq, dk, dv = A.backward(q, k, v, do, 0.4, False)
    o2, lse2 = A.forward(q, k[:, :, perm], v[:, :, perm], 0.4, False)
    dq2, dk2, dv2 = A.backward(q, k[:, :, perm], v[:, :, perm], do, 0.4, False)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dq2, dq, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk2, dk[:, :, perm], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv2, dv[:, :, perm], rtol=1e-11, atol=1e-12)
    o3, lse3 = A.forward(q[:, :, perm], k, v, 0.4, False)
    dq3, dk3, dv3 = A.backward(q[:, :, perm], k, v, do[:, :, perm], 0.4, False)
    np.testing.assert_allclose(o3, o[:, :, perm], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse3, lse[:, :, perm], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dq3, dq[:, :, perm], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk3, dk, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv3, dv, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_scale_reparametrisation(causal):
    """Only the product scale * Q enters the scores: Q -> c Q with scale -> scale / c
    leaves O, LSE, dK and dV unchanged and divides dQ by c."""
    n, d = 15, 5
    q, k, v, do = (rand(1, 2, n, d) for _ in range(4))
    c = 3.7
    o, lse = A.forward(q, k, v, 0.6, causal)
    o2, lse2 = A.forward(c * q, k, v, 0.6 / c, causal)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-12, atol=1e-13)
    dq, dk, dv = A.backward(q, k, v, do, 0.6, causal)
    dq2, dk2, dv2 = A.backward(c * q, k, v, do, 0.6 / c, causal)
    np.testing.assert_allclose(dq2, dq / c, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk2, dk, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv2, dv, rtol=1e-10, atol=1e-12)


def test_forward_rows_matches_forward():
    q, k, v = rand(1, 2, 40, 8), rand(1, 2, 40, 8), rand(1, 2, 40, 8)
    for causal in (False, True):
        o, lse = A.forward(q, k, v, 0.4, causal)
        rows = [0, 3, 17, 39]
        o_r, lse_r = A.forward_rows(q, k, v, 0.4, causal, 0, 1, rows)
        np.testing.assert_allclose(o_r, o[0, 1, rows], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse_r, lse[0, 1, rows], rtol=1e-13)


# ---------------------------------------------------------- brute force, pure Python


def _brute_force(q, k, v, do, scale, causal):
    """Scalar loops with math.exp: an implementation sharing nothing with numpy's."""
    n, d = len(q), len(q[0])
    o, lse, dq, dk, dv = [], [], [[0.0] * d for _ in range(n)], [[0.0] * d for _ in range(n)], [[0.0] * d for _ in range(n)]
    probs = []
    for i in range(n):
        js = range(i + 1) if causal else range(n)
        s = {j: scale * sum(q[i][c] * k[j][c] for c in range(d)) for j in js}
        mx = max(s.values())
        z = sum(math.exp(x - mx) for x in s.values())
        p = {j: math.exp(s[j] - mx) / z for j in js}
        probs.append(p)
        o.append([sum(p[j] * v[j][c] for j in js) for c in range(d)])
        lse.append(mx + math.log(z))
    for i in range(n):
        p = probs[i]
        di = sum(do[i][c] * o[i][c] for c in range(d))
        for j, pij in p.items():
            dpij = sum(do[i][c] * v[j][c] for c in range(d))
            dsij = pij * (dpij - di)
            for c in range(d):
                dv[j][c] += pij * do[i][c]
                dq[i][c] += scale * dsij * k[j][c]
                dk[j][c] += scale * dsij * q[i][c]
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_agreement(causal):
    n, d = 9, 4
    q, k, v, do = (rand(n, d) for _ in range(4))
    bo, blse, bdq, bdk, bdv = _brute_force(q.tolist(), k.tolist(), v.tolist(), do.tolist(), 0.45, causal)
    o, lse = A.forward(q[None, None], k[None, None], v[None, None], 0.45, causal)
    dq, dk, dv = A.backward(q[None, None], k[None, None], v[None, None], do[None, None], 0.45, causal)
    np.testing.assert_allclose(o[0, 0], bo, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], blse, rtol=1e-12)
    np.testing.assert_allclose(dq[0, 0], bdq, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk[0, 0], bdk, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv[0, 0], bdv, rtol=1e-11, atol=1e-12)


def test_torch_autograd_cross_check():
    """Library cross-check: torch fp64 autograd of softmax attention on tiny shapes."""
    torch = pytest.importorskip("torch")
    for causal in (False, True):
        n, d = 12, 6
        q, k, v, do = (rand(1, 2, n, d) for _ in range(4))
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        s = 0.6 * tq @ tk.transpose(-1, -2)
        if causal:
            s = s.masked_fill(~torch.ones(n, n, dtype=torch.bool).tril(), float("-inf"))
        o = torch.softmax(s, -1) @ tv
        lse = torch.logsumexp(s, -1)
        o.backward(torch.tensor(do))
        ro, rlse = A.forward(q, k, v, 0.6, causal)
        rdq, rdk, rdv = A.backward(q, k, v, do, 0.6, causal)
        np.testing.assert_allclose(ro, o.detach().numpy(), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(rlse, lse.detach().numpy(), rtol=1e-12)
        np.testing.assert_allclose(rdq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(rdk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(rdv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------- planted mistakes


def _mutant_backward(kind):
    def bwd(q, k, v, do, scale, causal):
        q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
        out = [np.empty_like(q), np.empty_like(k), np.empty_like(v)]
        for b in range(q.shape[0]):
            for h in range(q.shape[1]):
                p = A.probabilities(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], scale, causal)[0, 0]
                o = p @ v[b, h]
                dd = np.sum(do[b, h] * o, -1)
                dp = do[b, h] @ v[b, h].T
                ds = p * (dp - dd[:, None]) if kind != "sign" else p * (dd[:, None] - dp)
                dv = p.T @ do[b, h] if kind != "transpose" else p @ do[b, h]
                dq = (scale if kind != "dqnoscale" else 1.0) * ds @ k[b, h]
                dk = (scale if kind != "noscale" else 1.0) * ds.T @ q[b, h]
                out[0][b, h], out[1][b, h], out[2][b, h] = dq, dk, dv
        return tuple(out)
    return bwd


@pytest.mark.parametrize("kind", ["sign", "transpose", "noscale", "dqnoscale"])
def test_planted_mistakes_are_caught(kind):
    rng = np.random.default_rng(99)
    q, k, v, do = (rand(1, 1, 5, 3, rng=rng) for _ in range(4))
    errs = _fd_errors(q, k, v, do, 0.37, False, backward=_mutant_backward(kind))
    assert max(errs) > 1e-3, f"planted mistake '{kind}' slipped through: {errs}"


def test_reparametrisation_pin_catches_a_missing_dq_scale():
    """The scale reparametrisation pin, applied to a backward that forgets the scale
    on dQ only, fails (dQ would not scale by 1 / c)."""
    q, k, v, do = (rand(1, 1, 9, 4) for _ in range(4))
    bwd = _mutant_backward("dqnoscale")
    c = 3.7
    dq = bwd(q, k, v, do, 0.6, False)[0]
    dq2 = bwd(c * q, k, v, do, 0.6 / c, False)[0]
    assert not np.allclose(dq2, dq / c, rtol=1e-6, atol=1e-9)


def test_planted_causal_off_by_one_is_caught():
    """A strict mask (j < i) would leave row 0 empty; (j <= i+1) breaks causal row 0."""
    q, k, v = rand(1, 1, 6, 3), rand(1, 1, 6, 3), rand(1, 1, 6, 3)
    s = 0.5 * q[0, 0] @ k[0, 0].T
    wrong = np.where(np.arange(6)[None, :] <= np.arange(6)[:, None] + 1, s, -np.inf)
    p = np.exp(wrong - wrong.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    assert not np.allclose((p @ v[0, 0])[0], v[0, 0, 0])
    o, _ = A.forward(q, k, v, 0.5, True)
    np.testing.assert_array_equal(o[0, 0, 0], v[0, 0, 0])


# ------------------------------------------------------ row-restricted backward


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,block", [(37, 8), (64, 1024), (1, 4)])
def test_row_statistics_match_the_definition(causal, n, block):
    q, k, v, do = (rand(2, 2, n, 5) for _ in range(4))
    lse, dd = A.row_statistics(q, k, v, do, 0.45, causal, 1, 0, block=block)
    parts = A.backward_parts(q[1, 0], k[1, 0], v[1, 0], do[1, 0], 0.45, causal)
    np.testing.assert_allclose(lse, parts["LSE"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dd, parts["D"], rtol=1e-12, atol=1e-13)
    # D is also rowsum(P o dP), an identity independent of how O was formed.
    np.testing.assert_allclose(dd, np.sum(parts["P"] * parts["dP"], -1), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 5, 37, 130])
def test_backward_rows_match_backward(causal, n):
    rng = np.random.default_rng(n)
    q, k, v, do = (rand(2, 3, n, 6, rng=rng) for _ in range(4))
    k = k + 2.0  # a shifted key set, as in the long-sequence workload
    dq, dk, dv = A.backward(q, k, v, do, 0.41, causal)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, size=7)]))
    krows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, size=5)]))
    rq, rk, rv = A.backward_rows(q, k, v, do, 0.41, causal, 1, 2, rows, krows)
    np.testing.assert_allclose(rq, dq[1, 2, rows], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(rk, dk[1, 2, krows], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(rv, dv[1, 2, krows], rtol=1e-10, atol=1e-12)


def test_backward_rows_brute_force():
    n, d = 8, 3
    q, k, v, do = (rand(n, d) for _ in range(4))
    for causal in (False, True):
        _, _, bdq, bdk, bdv = _brute_force(q.tolist(), k.tolist(), v.tolist(), do.tolist(), 0.7, causal)
        rows = [0, 3, 7]
        rq, rk, rv = A.backward_rows(q[None, None], k[None, None], v[None, None], do[None, None], 0.7, causal,
                                     0, 0, rows, rows)
        np.testing.assert_allclose(rq, np.asarray(bdq)[rows], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(rk, np.asarray(bdk)[rows], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(rv, np.asarray(bdv)[rows], rtol=1e-11, atol=1e-12)


def _mutant_backward_rows(kind):
    """backward_rows with one planted mistake, for the pin below."""
    def bwd(q, k, v, do, scale, causal, b, h, qrows, krows):
        qh, kh, vh, doh = (np.asarray(x[b, h], dtype=np.float64) for x in (q, k, v, do))
        n = qh.shape[0]
        s_full = A.scores(qh, kh, scale, causal)
        m = np.max(s_full, -1)
        lse = m + np.log(np.sum(np.exp(s_full - m[:, None]), -1))
        if kind == "no_log_l":
            lse = m  # forgets the ln l term of the log-sum-exp
        p_full = np.exp(s_full - lse[:, None])
        dd = np.sum(doh * (p_full @ vh), -1)
        mask = A.visible_keys(n, causal)
        if kind == "mask_transposed":
            mask = mask.T
        st = np.where(mask[:, krows], scale * (qh @ kh[krows].T), -np.inf)
        pt = np.exp(st - lse[:, None])
        dst = pt * (doh @ vh[krows].T - dd[:, None])
        return None, scale * dst.T @ qh, pt.T @ doh
    return bwd


@pytest.mark.parametrize("kind", ["no_log_l", "mask_transposed"])
def test_backward_rows_planted_mistakes_are_caught(kind):
    q, k, v, do = (rand(1, 1, 12, 4) for _ in range(4))
    causal = kind == "mask_transposed"
    _, dk, dv = A.backward(q, k, v, do, 0.5, causal)
    rows = [0, 5, 11]
    _, mk, mv = _mutant_backward_rows(kind)(q, k, v, do, 0.5, causal, 0, 0, rows, rows)
    assert not (np.allclose(mk, dk[0, 0, rows], rtol=1e-6) and np.allclose(mv, dv[0, 0, rows], rtol=1e-6))
