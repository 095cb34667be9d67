"""Split-KV forward parity: fa_fwd_splitkv (through the C ABI) against the fp64 CPU oracle.

Each query block's key tiles are cut into parts; every part writes its own
normalised fp32 output and log-sum-exp, and a merge kernel combines them.  The
merged O and LSE must equal plain attention: partial softmax results combine
exactly through their maxima and sums ("ELI5: FlashAttention", softmax
statistics passage), so the oracle here is the same full-attention definition
the plain forward is held to.
"""

import numpy as np
import pytest

import oracle
from tiled_attention_tmem_gb300 import binding as b, inputs as I

from helpers import check_fwd, to_dev, to_f64

pytestmark = pytest.mark.gpu

# (B, H, N, d, causal, splits, sigma, scale)
CASES = [
    (1, 1, 1024, 128, False, 2, 1.0, None),
    # causal: in the later parts of a block its first query tile sees no key tile
    (1, 1, 1024, 128, True, 3, 1.0, None),
    # ragged tail, parts of a single key tile
    (1, 2, 333, 64, True, 4, 1.0, None),
    # more parts than key tiles (two): some work items have no key tile at all
    (1, 1, 200, 64, False, 5, 1.0, None),
    # 64-key tiles: a part holding only a block's last key tile is fully masked
    # for the block's first 64 rows (l = 0, weight 0 in the merge)
    (1, 1, 512, 256, True, 4, 0.5, 1.0 / 16),
    (1, 1, 300, 96, False, 3, 1.0, None),
    (1, 2, 384, 192, True, 3, 0.5, None),
    # a single row: one key tile, the second part empty
    (1, 1, 1, 64, False, 2, 1.0, None),
    (2, 1, 640, 256, False, 7, 1.0, None),
    (1, 1, 700, 384, True, 3, 1.0, None),
    (1, 1, 2048, 128, True, 16, 1.0, None),
    (1, 1, 4096, 64, False, 64, 1.0, None),
    # a large shift of the key means: partial maxima far apart across parts
    (1, 1, 1024, 128, False, 4, 1.0, None, 3.0),
]


def _run_split(x, B, H, N, d, scale, causal, splits):
    import torch
    from tiled_attention_tmem_gb300 import api
    q, k, v = (to_dev(t) for t in (x.q, x.k, x.v))
    o, lse = api.attention_forward(q, k, v, scale, causal, splits=splits)
    api.check_device_error()
    torch.cuda.synchronize()
    return o, lse


def _ids(c):
    return "b{}h{}n{}d{}{}s{}".format(*c[:4], "c" if c[4] else "", c[5]) + ("k" if len(c) > 8 else "")


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_split_forward_matches_oracle(case):
    B, H, N, d, causal, splits, sigma, scale = case[:8]
    shift = case[8] if len(case) > 8 else 0.0
    scale = scale if scale is not None else 1.0 / np.sqrt(d)
    x = I.make_inputs(B, H, N, d, seed=3000 + N + d + splits, sigma=sigma, k_shift=shift)
    o, lse = _run_split(x, B, H, N, d, scale, causal, splits)
    qf, kf, vf, _ = x.as_f64()
    o_ref, lse_ref = oracle.forward(qf, kf, vf, scale, causal)
    check_fwd(to_f64(o), to_f64(lse), o_ref, lse_ref, f"{case}")


def test_one_split_is_the_plain_forward():
    """splits = 1 takes no workspace and gives the plain kernel's bits."""
    import torch
    from tiled_attention_tmem_gb300 import api
    x = I.make_inputs(1, 2, 384, 128, seed=31)
    q, k, v = (to_dev(t) for t in (x.q, x.k, x.v))
    o1, l1 = api.attention_forward(q, k, v, 0.088, True)
    o2 = torch.empty_like(q)
    l2 = torch.empty_like(l1)
    st = b.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), l2.data_ptr(),
                          1, 2, 384, 128, 0.088, 1, 1, None, 0, torch.cuda.current_stream().cuda_stream)
    assert st == b.FA_OK
    api.check_device_error()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_forward_deterministic_and_close_to_plain():
    from tiled_attention_tmem_gb300 import api
    x = I.make_inputs(1, 1, 2048, 128, seed=32)
    a = _run_split(x, 1, 1, 2048, 128, 0.088, False, 4)
    c = _run_split(x, 1, 1, 2048, 128, 0.088, False, 4)
    assert np.array_equal(to_f64(a[0]), to_f64(c[0])) and np.array_equal(to_f64(a[1]), to_f64(c[1]))
    q, k, v = (to_dev(t) for t in (x.q, x.k, x.v))
    o, lse = api.attention_forward(q, k, v, 0.088, False)
    api.check_device_error()
    # Both are within the oracle tolerance; against each other they differ by
    # bf16 rounding of O (one ulp at |O| < 1) and fp32 rounding of the LSE.
    assert np.max(np.abs(to_f64(a[0]) - to_f64(o))) <= 8e-3
    assert np.max(np.abs(to_f64(a[1]) - to_f64(lse))) <= 1e-4


def test_chosen_splits_for_few_heads():
    """The cost model splits a long sequence of one head and leaves a full grid alone;
    its choice is run and checked on a shape where it splits."""
    assert b.fa_fwd_choose_splits(4, 16, 2048, 128, 1) == 1
    s = b.fa_fwd_choose_splits(1, 1, 4096, 128, 0)
    assert 2 <= s <= 16
    x = I.make_inputs(1, 1, 4096, 128, seed=33)
    o, lse = _run_split(x, 1, 1, 4096, 128, 128 ** -0.5, False, None)
    qf, kf, vf, _ = x.as_f64()
    o_ref, lse_ref = oracle.forward(qf, kf, vf, 128 ** -0.5, False)
    check_fwd(to_f64(o), to_f64(lse), o_ref, lse_ref, f"auto splits={s}")


def test_split_full_size_sampled_rows():
    """A long single-head sequence at the split count the cost model picks, checked
    on sampled rows the oracle computes one by one."""
    import torch
    from tiled_attention_tmem_gb300 import api
    B, H, N, d = 1, 1, 16384, 128
    x = I.make_inputs(B, H, N, d, seed=34)
    q, k, v = (to_dev(t) for t in (x.q, x.k, x.v))
    s = b.fa_fwd_choose_splits(B, H, N, d, 1)
    assert s > 1
    o, lse = api.attention_forward(q, k, v, d ** -0.5, True, splits=s)
    api.check_device_error()
    torch.cuda.synchronize()
    qf, kf, vf, _ = x.as_f64()
    rng = np.random.default_rng(35)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], rng.integers(0, N, 24)]))
    o_ref, lse_ref = oracle.forward_rows(qf, kf, vf, d ** -0.5, True, 0, 0, rows)
    check_fwd(to_f64(o)[0, 0, rows], to_f64(lse)[0, 0, rows], o_ref, lse_ref, f"N={N} splits={s}")
