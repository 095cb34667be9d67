"""Plain fp64 scaled-dot-product attention: the definition the tiled method must reproduce.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

What is computed, and where it comes from
-----------------------------------------
"ELI5: FlashAttention" (Gordić), the passages on tiling and on the softmax
statistics, states that chopping the softmax into blocks still yields precisely
the same result as the direct computation.  The oracle is therefore the direct
computation, for every (batch, head) separately:

    s_ij  = scale * sum_c Q_ic K_jc                      for j in J(i)
    m_i   = max_j s_ij,   l_i = sum_j exp(s_ij - m_i)
    P_ij  = exp(s_ij - m_i) / l_i   (0 for j not in J(i))
    O_i   = sum_j P_ij V_j
    LSE_i = m_i + ln l_i            (natural log of sum_j exp(s_ij))

J(i) = {0..N-1} without a mask and {0..i} with the causal ("triangular") mask
mentioned in the Hacker News thread on FlashAttention's hardware dependence.

The backward uses the operand list of the issue thread "Potential algorithmic
improvements for backward pass" (Q, K, V, O, log-sum-exp, dO, dV, dK, dQ) and the
standard softmax-attention gradients:

    D_i   = sum_c dO_ic O_ic
    dP_ij = sum_c dO_ic V_jc
    dS_ij = P_ij (dP_ij - D_i)
    dV_j  = sum_i P_ij dO_i
    dQ_i  = scale * sum_j dS_ij K_j
    dK_j  = scale * sum_i dS_ij Q_i

Readings where the pages are silent: LSE is the natural log of the sum of
exponentials of the *scaled* scores; the scale multiplies the fp64 scores (it
is not folded into a rounded Q); dQ and dK include the scale.

Arrays are [B, H, N, d] (LSE and D are [B, H, N]); all arithmetic is fp64.  A
matrix product (numpy ``@``) is used as a library primitive; S, P, dP and dS
are materialised in full for each head, one head at a time.
"""

from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def visible_keys(n: int, causal: bool) -> np.ndarray:
    """Boolean [n, n] matrix: entry (i, j) is True when query i may attend to key j.

    Causal reading: key j is visible to query i exactly when j <= i, so every row
    keeps at least one key.
    """
    if causal:
        return np.tril(np.ones((n, n), dtype=bool))
    return np.ones((n, n), dtype=bool)


def scores(q, k, scale: float, causal: bool) -> np.ndarray:
    """Scaled scores s = scale * Q K^T per head, -inf where the key is masked."""
    q = _f64(q)
    k = _f64(k)
    s = scale * (q @ np.swapaxes(k, -1, -2))
    if causal:
        n = q.shape[-2]
        s = np.where(visible_keys(n, True), s, -np.inf)
    return s


def _softmax_stats(s: np.ndarray):
    """Row max m, exp-sum l and probabilities P of a score block with -inf masks."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)  # exp(-inf) = 0 for masked keys
    l = np.sum(e, axis=-1, keepdims=True)
    return m, l, e / l


def probabilities(q, k, scale: float, causal: bool) -> np.ndarray:
    """Softmax probabilities P [B, H, N, N] (rows sum to one; masked entries are 0)."""
    _, _, p = _softmax_stats(scores(q, k, scale, causal))
    return p


def forward(q, k, v, scale: float, causal: bool):
    """Returns (O [B,H,N,d], LSE [B,H,N]) in fp64, one head at a time."""
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    b_, h_, n, d = q.shape
    o = np.empty((b_, h_, n, v.shape[-1]), dtype=np.float64)
    lse = np.empty((b_, h_, n), dtype=np.float64)
    for b in range(b_):
        for h in range(h_):
            s = scores(q[b, h], k[b, h], scale, causal)
            m, l, p = _softmax_stats(s)
            o[b, h] = p @ v[b, h]
            lse[b, h] = (m + np.log(l))[:, 0]
    return o, lse


def forward_rows(q, k, v, scale: float, causal: bool, b: int, h: int, rows):
    """O and LSE of selected query rows of one head (rows are independent).

    Used on full-size inputs where only a sample of rows is checked.  Each row is
    the same definition as ``forward`` restricted to that row.
    """
    qh = _f64(q[b, h])
    kh = _f64(k[b, h])
    vh = _f64(v[b, h])
    rows = np.asarray(rows, dtype=np.int64)
    s = scale * (qh[rows] @ kh.T)
    if causal:
        cols = np.arange(kh.shape[0])[None, :]
        s = np.where(cols <= rows[:, None], s, -np.inf)
    m, l, p = _softmax_stats(s)
    return p @ vh, (m + np.log(l))[:, 0]


def backward_parts(q, k, v, do, scale: float, causal: bool):
    """Every intermediate of the backward for ONE head ([N, d] inputs).

    Returns a dict with S, P, O, LSE, D, dP, dS, dQ, dK, dV (fp64).  The
    recomputation of P from the forward's statistics (the "recomputation" idea
    of the ELI5 article) is mathematically the same P, so the oracle simply
    evaluates the definition again.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    do = _f64(do)
    s = scores(q, k, scale, causal)
    m, l, p = _softmax_stats(s)
    o = p @ v
    lse = (m + np.log(l))[:, 0]
    dd = np.sum(do * o, axis=-1)
    dp = do @ v.T
    ds = p * (dp - dd[:, None])
    dv = p.T @ do
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return {
        "S": s, "P": p, "O": o, "LSE": lse, "D": dd,
        "dP": dp, "dS": ds, "dQ": dq, "dK": dk, "dV": dv,
    }


def backward(q, k, v, do, scale: float, causal: bool):
    """Returns (dQ, dK, dV) [B,H,N,d] fp64 from the oracle's own fp64 O and P."""
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    do = _f64(do)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            parts = backward_parts(q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
            dq[b, h] = parts["dQ"]
            dk[b, h] = parts["dK"]
            dv[b, h] = parts["dV"]
    return dq, dk, dv


def row_statistics(q, k, v, do, scale: float, causal: bool, b: int, h: int, block: int = 256):
    """LSE_i and D_i of every query row of one head, each from its own full score row.

    LSE_i = m_i + ln l_i over the visible keys of row i (the forward's per-row
    statistic that the backward recomputes P from, "ELI5: FlashAttention",
    recomputation passage) and D_i = sum_c dO_ic O_ic with O_i = sum_j P_ij V_j.
    Every row is the definition applied to that row alone; rows are taken
    ``block`` at a time only to bound memory at long sequences.
    """
    qh, kh, vh, doh = (_f64(x[b, h]) for x in (q, k, v, do))
    n = qh.shape[0]
    lse = np.empty(n, dtype=np.float64)
    dd = np.empty(n, dtype=np.float64)
    cols = np.arange(kh.shape[0])[None, :]
    for r0 in range(0, n, block):
        rows = np.arange(r0, min(n, r0 + block))
        s = scale * (qh[rows] @ kh.T)
        if causal:
            s = np.where(cols <= rows[:, None], s, -np.inf)
        m, l, p = _softmax_stats(s)
        lse[rows] = (m + np.log(l))[:, 0]
        dd[rows] = np.sum(doh[rows] * (p @ vh), axis=-1)
    return lse, dd


def backward_rows(q, k, v, do, scale: float, causal: bool, b: int, h: int, qrows, krows):
    """dQ of chosen query rows and dK, dV of chosen key rows of one head.

    For sequences too long for ``backward_parts``' N x N matrices.  With the
    per-row statistics of ``row_statistics`` (LSE_i, D_i for every row i):

        P_ij  = exp(s_ij - LSE_i)  (0 where key j is masked for query i)
        dS_ij = P_ij (dO_i . V_j - D_i)
        dQ_i  = scale * sum_j dS_ij K_j        for i in qrows (row i of P, dS)
        dV_j  = sum_i P_ij dO_i                for j in krows (column j of P)
        dK_j  = scale * sum_i dS_ij Q_i        for j in krows (column j of dS)

    the same gradients as ``backward``, restricted to the chosen rows.
    Returns (dQ [len(qrows), d], dK [len(krows), d], dV [len(krows), d]).
    """
    qh, kh, vh, doh = (_f64(x[b, h]) for x in (q, k, v, do))
    n = qh.shape[0]
    lse, dd = row_statistics(q, k, v, do, scale, causal, b, h)
    qrows = np.asarray(qrows, dtype=np.int64)
    krows = np.asarray(krows, dtype=np.int64)
    # Rows of P and dS: query i against every key.
    s = scale * (qh[qrows] @ kh.T)
    if causal:
        s = np.where(np.arange(n)[None, :] <= qrows[:, None], s, -np.inf)
    p = np.exp(s - lse[qrows, None])
    ds = p * (doh[qrows] @ vh.T - dd[qrows, None])
    dq = scale * (ds @ kh)
    # Columns of P and dS: every query i against key j.
    st = scale * (qh @ kh[krows].T)
    if causal:
        st = np.where(krows[None, :] <= np.arange(n)[:, None], st, -np.inf)
    pt = np.exp(st - lse[:, None])
    dst = pt * (doh @ vh[krows].T - dd[:, None])
    dv = pt.T @ doh
    dk = scale * (dst.T @ qh)
    return dq, dk, dv
