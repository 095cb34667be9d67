"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (code inside an allocator, a memory-capped plugin host, a runtime
that only hands out input and output buffers) cannot provide fa_bwd's
workspace.  fa_bwd_noalloc keeps its scratch in a static device array inside
the library instead.  These tests call it through the C ABI twice in a row and
compare each result with the workspace-taking fa_bwd on the same inputs and with
the fp64 CPU oracle, within the gradient tolerance used by the other backward
tests; they also check that an expired in-kernel wait on this path is reported
through its own allocation-free status call.  The file is named so that pytest
collects it last.
"""

import numpy as np
import pytest

from tiled_attention_tmem_gb300 import binding as b
from tiled_attention_tmem_gb300 import inputs as I

import oracle

from helpers import TOL_GRAD_REL, check_grads, to_dev, to_f64

pytestmark = pytest.mark.gpu

CASES = [
    # (B, H, N, d, causal, variant)
    (1, 2, 384, 128, True, b.FA_BWD_5GEMM),
    (1, 2, 384, 128, True, b.FA_BWD_7GEMM),
    (2, 2, 200, 64, False, b.FA_BWD_AUTO),
    (1, 2, 256, 256, True, b.FA_BWD_7GEMM),
    # head dims run on zero-padded tiles
    (1, 2, 300, 96, True, b.FA_BWD_5GEMM),
    (1, 2, 200, 192, False, b.FA_BWD_AUTO),
    (1, 2, 300, 384, True, b.FA_BWD_AUTO),
]


def _inputs(B, H, N, d, causal):
    import torch
    from tiled_attention_tmem_gb300 import api
    x = I.make_inputs(B, H, N, d, seed=4242 + N + d)
    q, k, v, do = (to_dev(t) for t in (x.q, x.k, x.v, x.do))
    scale = 1.0 / np.sqrt(d)
    o, lse = api.attention_forward(q, k, v, scale, causal)
    torch.cuda.synchronize()
    return q, k, v, o, do, lse, scale


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}n{}d{}{}-v{}".format(*c[:4], "c" if c[4] else "", c[5]))
def test_noalloc_matches_workspace_backward_twice(case):
    import torch
    from tiled_attention_tmem_gb300 import api
    B, H, N, d, causal, variant = case
    q, k, v, o, do, lse, scale = _inputs(B, H, N, d, causal)
    ref = [to_f64(t) for t in api.attention_backward(q, k, v, o, do, lse, scale, causal, variant=variant)]
    api.check_device_error()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        for t in (dq, dk, dv):
            t.fill_(float("nan"))  # every element must be written by the call
        st = b.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                              lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                              B, H, N, d, scale, int(causal), variant, stream)
        assert st == b.FA_OK, b.fa_strerror(st)
        torch.cuda.synchronize()
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            g = to_f64(got)
            assert np.all(np.isfinite(g)), f"call {call}: {name} has unwritten or non-finite entries"
            err = float(np.max(np.abs(g - want)))
            assert err <= TOL_GRAD_REL * float(np.max(np.abs(want))), f"call {call}: {name} err {err}"


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    # 5-GEMM for B*H = 1024, N = 2048, d = 128 needs about 1.1 GB of scratch.
    A = 1 << 20  # aligned placeholder address; nothing is launched or dereferenced
    st = b.fa_bwd_noalloc(A, A, A, A, A, A, A, A, A, 64, 16, 2048, 128, 0.088, 1, b.FA_BWD_5GEMM, None)
    assert st == b.FA_ERR_WORKSPACE
    # 7-GEMM needs only the row statistics (8 bytes per padded row): 64 MiB covers 8 Mi rows.
    st = b.fa_bwd_noalloc(A, A, A, A, A, A, A, A, A, 1024, 64, 16384, 128, 0.088, 1, b.FA_BWD_7GEMM, None)
    assert st == b.FA_ERR_WORKSPACE


def _noalloc(q, k, v, o, do, lse, B, H, N, d, scale, causal, variant):
    import torch
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for t in (dq, dk, dv):
        t.fill_(float("nan"))
    stream = torch.cuda.current_stream().cuda_stream
    st = b.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                          lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                          B, H, N, d, scale, int(causal), variant, stream)
    assert st == b.FA_OK, b.fa_strerror(st)
    status, site = b.fa_bwd_noalloc_device_error(stream)
    assert status == b.FA_OK, (status, hex(site))
    return dq, dk, dv


@pytest.mark.parametrize("variant", [b.FA_BWD_5GEMM, b.FA_BWD_7GEMM])
def test_noalloc_matches_the_oracle_twice(variant):
    B, H, N, d, causal = 1, 2, 333, 128, True
    q, k, v, o, do, lse, scale = _inputs(B, H, N, d, causal)
    x = I.make_inputs(B, H, N, d, seed=4242 + N + d)
    qf, kf, vf, dof = x.as_f64()
    ref = oracle.backward(qf, kf, vf, dof, scale, causal)
    for call in range(2):
        got = _noalloc(q, k, v, o, do, lse, B, H, N, d, scale, causal, variant)
        check_grads([to_f64(t) for t in got], ref, f"no-alloc call {call}")


def test_noalloc_auto_falls_back_to_seven_gemm_beyond_the_array():
    """B*H = 64, N = 2048, d = 128: the 5-GEMM scratch (68 MB) exceeds the 64 MiB
    array, so AUTO runs the 7-GEMM form; it must match fa_bwd's 7-GEMM result bit
    for bit (the 7-GEMM form is deterministic) and the oracle on sampled heads."""
    from tiled_attention_tmem_gb300 import api
    B, H, N, d, causal = 1, 64, 2048, 128, True
    assert b.fa_bwd_workspace_size(B, H, N, d, b.FA_BWD_5GEMM) > b.FA_NOALLOC_SCRATCH_BYTES
    q, k, v, o, do, lse, scale = _inputs(B, H, N, d, causal)
    want = [to_f64(t) for t in api.attention_backward(q, k, v, o, do, lse, scale, causal,
                                                      variant=b.FA_BWD_7GEMM)]
    api.check_device_error()
    got = [to_f64(t) for t in _noalloc(q, k, v, o, do, lse, B, H, N, d, scale, causal, b.FA_BWD_AUTO)]
    for g, w in zip(got, want):
        assert np.array_equal(g, w)
    x = I.make_inputs(B, H, N, d, seed=4242 + N + d)
    for h in (0, H - 1):
        qf, kf, vf, dof = (I.bf16_bits_to_f64(t[:, h:h + 1]) for t in (x.q, x.k, x.v, x.do))
        ref = oracle.backward(qf, kf, vf, dof, scale, causal)
        check_grads([t[:, h:h + 1] for t in got], ref, f"no-alloc AUTO head {h}")


def test_noalloc_timeout_is_reported_by_its_own_status_call():
    """An expired bounded wait on the no-alloc path (the library's self-test warp,
    waiting on a barrier nothing completes) is reported by
    fa_bwd_noalloc_device_error, cleared by reading it, and the next call computes."""
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    assert b.fa_bwd_noalloc_device_error(stream)[0] == b.FA_OK
    assert b.fa_bwd_noalloc_watchdog_selftest(stream) == b.FA_OK
    status, site = b.fa_bwd_noalloc_device_error(stream)
    assert status == b.FA_ERR_DEVICE_TIMEOUT and site == (6 << 8) | 1
    assert b.fa_bwd_noalloc_device_error(stream)[0] == b.FA_OK
    # The workspace entry points' error word was not touched.
    assert b.fa_get_device_error(stream)[0] == b.FA_OK
    B, H, N, d, causal = 1, 2, 256, 64, False
    q, k, v, o, do, lse, scale = _inputs(B, H, N, d, causal)
    x = I.make_inputs(B, H, N, d, seed=4242 + N + d)
    qf, kf, vf, dof = x.as_f64()
    got = _noalloc(q, k, v, o, do, lse, B, H, N, d, scale, causal, b.FA_BWD_AUTO)
    check_grads([to_f64(t) for t in got], oracle.backward(qf, kf, vf, dof, scale, causal), "after timeout")
