"""Blockwise ("online") softmax merge in fp64, as the tiled method performs it.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"ELI5: FlashAttention" (Gordić), the passage on the two statistics: the scores
of a row are processed block by block; each block contributes its maximum m(x)
and its sum of exponentials l(x), and partial results are fused with the
normalising coefficients exp(m_old - m_new) so that the final softmax is exactly
the direct one.  This module restates that algorithm, in the article's order, so
the tests can check it against the direct definition in ``attention``:

    for each key block B:
        m_B = max_{j in B} s_ij            (masked keys are -inf)
        p_j = exp(s_ij - m_B),  l_B = sum_j p_j,  o_B = sum_j p_j V_j
        m'  = max(m, m_B)
        l   = exp(m - m') l + exp(m_B - m') l_B
        o   = exp(m - m') o + exp(m_B - m') o_B
        m   = m'
    O = o / l,  LSE = m + ln l

Blocks that are entirely masked for a row leave that row's statistics untouched.
"""

from __future__ import annotations

import numpy as np


def merge_partials(m_a, l_a, o_a, m_b, l_b, o_b):
    """Fuse two partial softmax results of the same rows (m: [R], l: [R], o: [R, d])."""
    m_a = np.asarray(m_a, dtype=np.float64)
    m_b = np.asarray(m_b, dtype=np.float64)
    m = np.maximum(m_a, m_b)
    # A side with no visible key has m = -inf and contributes nothing.
    fa = np.where(np.isneginf(m_a), 0.0, np.exp(np.where(np.isneginf(m_a), 0.0, m_a - m)))
    fb = np.where(np.isneginf(m_b), 0.0, np.exp(np.where(np.isneginf(m_b), 0.0, m_b - m)))
    l = fa * l_a + fb * l_b
    o = fa[:, None] * o_a + fb[:, None] * o_b
    return m, l, o


def blockwise_forward(q, k, v, scale: float, causal: bool, block_sizes):
    """O and LSE of ONE head ([N, d] inputs) by merging key blocks of the given sizes.

    ``block_sizes`` lists consecutive block lengths that must add up to N.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_q = q.shape[0]
    n_k = k.shape[0]
    if sum(block_sizes) != n_k:
        raise ValueError("block sizes must cover every key exactly once")
    m = np.full(n_q, -np.inf)
    l = np.zeros(n_q)
    o = np.zeros((n_q, v.shape[1]))
    rows = np.arange(n_q)[:, None]
    start = 0
    for size in block_sizes:
        cols = np.arange(start, start + size)[None, :]
        s = scale * (q @ k[start:start + size].T)
        if causal:
            s = np.where(cols <= rows, s, -np.inf)
        m_blk = np.max(s, axis=1)
        safe = np.where(np.isneginf(m_blk), 0.0, m_blk)
        p = np.exp(s - safe[:, None])
        l_blk = np.sum(p, axis=1)
        o_blk = p @ v[start:start + size]
        m, l, o = merge_partials(m, l, o, m_blk, l_blk, o_blk)
        start += size
    return o / l[:, None], m + np.log(l)


def split_forward(q, k, v, scale: float, causal: bool, part_sizes):
    """O and LSE of ONE head ([N, d] inputs) by the split-KV route, in fp64.

    The same statistics merge as above, taken over whole key ranges instead of
    running block by block ("ELI5: FlashAttention", softmax statistics passage):
    each consecutive key range ("part") s of ``part_sizes`` is finished on its
    own into a normalised output and its log-sum-exp,

        O_s = sum_{j in s} exp(s_ij - L_s) V_j,   L_s = ln sum_{j in s} exp(s_ij)

    (L_s = -inf and O_s = 0 where no key of the part is visible to the row), and
    the parts are combined with the log-sum-exp weights

        L = ln sum_s exp(L_s),   O = sum_s exp(L_s - L) O_s.

    A part of size 0 is allowed and contributes nothing.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_q = q.shape[0]
    n_k = k.shape[0]
    if sum(part_sizes) != n_k or min(part_sizes, default=0) < 0:
        raise ValueError("part sizes must cover every key exactly once")
    rows = np.arange(n_q)[:, None]
    o_parts, l_parts = [], []
    start = 0
    for size in part_sizes:
        cols = np.arange(start, start + size)[None, :]
        s = scale * (q @ k[start:start + size].T)
        if causal:
            s = np.where(cols <= rows, s, -np.inf)
        if size == 0:
            m_s = np.full(n_q, -np.inf)
        else:
            m_s = np.max(s, axis=1)
        seen = ~np.isneginf(m_s)
        safe = np.where(seen, m_s, 0.0)
        p = np.exp(s - safe[:, None]) if size else np.zeros((n_q, 0))
        l_s = np.sum(p, axis=1)
        o_s = np.zeros((n_q, v.shape[1]))
        o_s[seen] = (p @ v[start:start + size])[seen] / l_s[seen][:, None]
        lse_s = np.where(seen, safe + np.log(np.where(seen, l_s, 1.0)), -np.inf)
        o_parts.append(o_s)
        l_parts.append(lse_s)
        start += size
    lse_parts = np.stack(l_parts)           # [S, R]
    top = np.max(lse_parts, axis=0)         # every row sees at least one key overall
    w = np.where(np.isneginf(lse_parts), 0.0, np.exp(lse_parts - top[None, :]))
    total = np.sum(w, axis=0)
    lse = top + np.log(total)
    o = np.einsum("sr,srd->rd", w / total[None, :], np.stack(o_parts))
    return o, lse
