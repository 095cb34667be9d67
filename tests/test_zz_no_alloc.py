"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (code inside an allocator, a memory-capped plugin host, a runtime
that only hands out input and output buffers) cannot provide fa_bwd's
workspace.  fa_bwd_noalloc keeps its scratch in a static device array inside
the library instead.  These tests call it through the C ABI twice in a row and
compare each result with the workspace-taking fa_bwd on the same inputs, within
the gradient tolerance used by the other backward tests.  The file is named so
that pytest collects it last.
"""

import numpy as np
import pytest

from tiled_attention_tmem_gb300 import binding as b
from tiled_attention_tmem_gb300 import inputs as I

from helpers import TOL_GRAD_REL, to_dev, to_f64

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
