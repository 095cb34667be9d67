"""Host-side checks of the torch convenience layer (no GPU): tensors that are not
contiguous CUDA tensors of the right dtype and shape are rejected before the
library is called."""

import pytest
import torch

from tiled_attention_tmem_gb300 import api


def _bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def test_forward_rejects_host_tensors():
    q = _bf16(1, 2, 128, 64)
    with pytest.raises(ValueError, match="contiguous CUDA"):
        api.attention_forward(q, q, q)


def test_backward_rejects_host_tensors():
    q = _bf16(1, 2, 128, 64)
    lse = torch.zeros((1, 2, 128), dtype=torch.float32)
    with pytest.raises(ValueError, match="contiguous CUDA"):
        api.attention_backward(q, q, q, q, q, lse)


def test_forward_rejects_wrong_dtype_before_anything_else():
    q = torch.zeros((1, 2, 128, 64), dtype=torch.float16)
    with pytest.raises(ValueError, match="bfloat16"):
        api.attention_forward(q, q, q)


def test_split_workspace_size_matches_the_layout():
    # fp32 parts [S, B, H, N, d] then fp32 part LSEs [S, B, H, N], each 256-byte aligned
    s, B, H, N, d = 3, 2, 2, 200, 128
    parts = 4 * s * B * H * N * d
    lses = 4 * s * B * H * N
    r = lambda x: (x + 255) // 256 * 256
    assert api.splitkv_workspace_bytes(B, H, N, d, s) == r(parts) + r(lses)
    assert api.splitkv_workspace_bytes(B, H, N, d, 1) == 0


def test_forward_rejects_wrong_shapes():
    q = _bf16(1, 2, 128, 64)
    with pytest.raises(ValueError, match="shape"):
        api.attention_forward(q, _bf16(1, 2, 64, 64), q)
    with pytest.raises(ValueError, match="shape"):
        api.attention_forward(_bf16(2, 128, 64), q, q)


def test_forward_rejects_a_wrong_out_or_lse():
    q = _bf16(1, 2, 128, 64)
    with pytest.raises(ValueError, match="out must have shape"):
        api.attention_forward(q, q, q, out=_bf16(1, 2, 128, 32))
    with pytest.raises(ValueError, match="lse must be"):
        api.attention_forward(q, q, q, lse=torch.zeros((1, 2, 128), dtype=torch.float64))
    with pytest.raises(ValueError, match="lse must have shape"):
        api.attention_forward(q, q, q, lse=torch.zeros((1, 2, 64), dtype=torch.float32))


def test_backward_rejects_wrong_shapes():
    q = _bf16(1, 2, 128, 64)
    lse = torch.zeros((1, 2, 128), dtype=torch.float32)
    with pytest.raises(ValueError, match="do must have shape"):
        api.attention_backward(q, q, q, q, _bf16(1, 2, 128, 32), lse)
    with pytest.raises(ValueError, match="lse must have shape"):
        api.attention_backward(q, q, q, q, q, torch.zeros((1, 2, 127), dtype=torch.float32))
    with pytest.raises(ValueError, match="lse must be"):
        api.attention_backward(q, q, q, q, q, torch.zeros((1, 2, 128), dtype=torch.float16))


def test_backward_rejects_wrong_grads_and_workspace():
    q = _bf16(1, 2, 128, 64)
    lse = torch.zeros((1, 2, 128), dtype=torch.float32)
    with pytest.raises(ValueError, match="dk must have shape"):
        api.attention_backward(q, q, q, q, q, lse, grads=(q, _bf16(1, 2, 128, 16), q))
    with pytest.raises(ValueError, match="grads must be"):
        api.attention_backward(q, q, q, q, q, lse, grads=(q, q))
    with pytest.raises(ValueError, match="workspace must be"):
        api.attention_backward(q, q, q, q, q, lse, workspace=torch.zeros(16, dtype=torch.float32))
