"""Concurrency through the C ABI: calls on two streams at once, and a CUDA graph of fwd + bwd.

The kernels are launched with programmatic stream serialization and the 5-GEMM kernel claims
its work from a counter in the caller's workspace, so these check that neither leaks across
streams or breaks under graph capture.  References are the same calls made one after another
on the default stream: the forward and the 7-GEMM backward are bitwise reproducible, the
5-GEMM dQ (reduced in nondeterministic order) is compared within its tolerance.
"""

import numpy as np
import pytest

from tiled_attention_tmem_gb300 import binding as b, inputs as I

from helpers import TOL_GRAD_REL, to_dev

pytestmark = pytest.mark.gpu

PROBLEMS = [
    # (B, H, N, d, causal, seed); the last is one head of 2048 rows, where the backward
    # splits the dK/dV kernel's query ranges (and, 7-GEMM, the dQ kernel's key ranges)
    # with partial sums in the caller's workspace
    (2, 4, 1024, 128, True, 31),
    (1, 8, 768, 64, False, 32),
    (1, 1, 2048, 128, True, 35),
]


def _inputs(B, H, N, d, seed):
    x = I.make_inputs(B, H, N, d, seed=seed)
    return tuple(to_dev(t) for t in (x.q, x.k, x.v, x.do))


def _run(tensors, causal, variant, stream=None):
    from tiled_attention_tmem_gb300 import api
    q, k, v, do = tensors
    o, lse = api.attention_forward(q, k, v, None, causal, stream=stream)
    grads = api.attention_backward(q, k, v, o, do, lse, None, causal, variant=variant, stream=stream)
    return (o, lse) + tuple(grads)


def _compare(got, ref, variant):
    import torch
    names = ("o", "lse", "dq", "dk", "dv")
    for name, g, r in zip(names, got, ref):
        if name == "dq" and variant == b.FA_BWD_5GEMM:
            err = (g.float() - r.float()).abs().max().item()
            assert err <= TOL_GRAD_REL * r.float().abs().max().item(), f"{name}: {err}"
        else:
            assert torch.equal(g, r), f"{name} differs"


@pytest.mark.parametrize("variant", [b.FA_BWD_5GEMM, b.FA_BWD_7GEMM])
def test_two_streams_concurrently(variant):
    import torch
    from tiled_attention_tmem_gb300 import api
    data = [_inputs(B, H, N, d, seed) for B, H, N, d, _, seed in PROBLEMS]
    refs = [_run(t, p[4], variant) for t, p in zip(data, PROBLEMS)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in PROBLEMS]
    outs = []
    for rep in range(3):
        outs = []
        for t, p, s in zip(data, PROBLEMS, streams):
            with torch.cuda.stream(s):
                outs.append(_run(t, p[4], variant, stream=s.cuda_stream))
        torch.cuda.synchronize()
        for o, r in zip(outs, refs):
            _compare(o, r, variant)
    api.check_device_error()


GRAPH_PROBLEMS = [
    # (B, H, N, d, causal, seed, splits): the bench-like shape, one long head with the split-KV
    # forward and the query-split backward (extra merge and sum kernels), and head dim 384
    (2, 4, 1024, 128, True, 31, 1),
    (1, 1, 4096, 128, True, 33, 4),
    (1, 2, 640, 384, True, 34, 1),
]


@pytest.mark.parametrize("problem", GRAPH_PROBLEMS, ids=lambda p: "b{}h{}n{}d{}".format(*p[:4]))
def test_cuda_graph_replay(problem):
    import torch
    from tiled_attention_tmem_gb300 import api
    B, H, N, d, causal, seed, splits = problem
    q, k, v, do = _inputs(B, H, N, d, seed)
    variant = b.FA_BWD_7GEMM
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    ws = torch.empty(b.fa_bwd_workspace_size(B, H, N, d, variant), dtype=torch.uint8, device=q.device)

    split_ws = torch.empty(max(1, b.fa_fwd_splitkv_workspace_size(B, H, N, d, splits)), dtype=torch.uint8,
                           device=q.device)

    def step():
        api.attention_forward(q, k, v, None, causal, out=o, lse=lse, splits=splits, workspace=split_ws)
        api.attention_backward(q, k, v, o, do, lse, None, causal, variant=variant, workspace=ws, grads=grads)

    step()  # eager first: creates the library's device state outside the capture
    torch.cuda.synchronize()
    ref = tuple(t.clone() for t in (o, lse) + grads)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step()
    torch.cuda.synchronize()
    for t in (o, lse) + grads:
        t.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for g, r in zip((o, lse) + grads, ref):
        assert torch.equal(g, r)
    api.check_device_error()
