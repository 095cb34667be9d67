"""Torch-tensor convenience wrappers over the C ABI (marshalling only).

PyTorch supplies device memory and the current stream; the computation runs in
the CUDA library through ``binding``.  Tensors must be CUDA, bf16 (LSE fp32),
C-contiguous and shaped [B, H, N, d].
"""

from __future__ import annotations

import math

from . import binding as _b


def _check(t, name, dtype):
    import torch
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    return t


def _stream(stream):
    import torch
    return stream if stream is not None else torch.cuda.current_stream().cuda_stream


def attention_forward(q, k, v, scale: float | None = None, causal: bool = False,
                      out=None, lse=None, stream=None, splits: int | None = 1, workspace=None):
    """Returns (O bf16 [B,H,N,d], LSE fp32 [B,H,N]).

    ``splits`` > 1 runs the split-KV form (``fa_fwd_splitkv``) with that many key
    parts per query block; ``None`` takes ``fa_fwd_choose_splits``.  ``workspace``
    (a uint8 CUDA tensor of ``splitkv_workspace_bytes`` or more) is allocated when
    needed and not given."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16)
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if out is None else _check(out, "out", torch.bfloat16)
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if splits is None:
        splits = _b.fa_fwd_choose_splits(B, H, N, d, int(causal))
    if splits == 1:
        st = _b.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                       B, H, N, d, scale, int(causal), _stream(stream))
        if st != _b.FA_OK:
            raise _b.FaError(st, "fa_fwd")
        return o, l
    if workspace is None:
        need = _b.fa_fwd_splitkv_workspace_size(B, H, N, d, splits)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = _b.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                           B, H, N, d, scale, int(causal), splits, workspace.data_ptr(),
                           workspace.numel(), _stream(stream))
    if st != _b.FA_OK:
        raise _b.FaError(st, "fa_fwd_splitkv")
    return o, l


def splitkv_workspace_bytes(B, H, N, d, splits) -> int:
    return _b.fa_fwd_splitkv_workspace_size(B, H, N, d, splits)


def workspace_bytes(B, H, N, d, variant=_b.FA_BWD_AUTO) -> int:
    return _b.fa_bwd_workspace_size(B, H, N, d, variant)


def attention_backward(q, k, v, o, do, lse, scale: float | None = None, causal: bool = False,
                       variant: int = _b.FA_BWD_AUTO, workspace=None, grads=None, stream=None):
    """Returns (dQ, dK, dV) bf16 [B,H,N,d]; ``workspace`` is a uint8 CUDA tensor or None."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _check(t, n, torch.bfloat16)
    _check(lse, "lse", torch.float32)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    need = _b.fa_bwd_workspace_size(B, H, N, d, variant)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    dq, dk, dv = grads
    st = _b.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                   lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                   B, H, N, d, scale, int(causal), variant,
                   workspace.data_ptr(), workspace.numel(), _stream(stream))
    if st != _b.FA_OK:
        raise _b.FaError(st, "fa_bwd")
    return dq, dk, dv


def check_device_error(stream=None):
    """Synchronises the stream and raises if a bounded in-kernel wait expired."""
    st, site = _b.fa_get_device_error(_stream(stream))
    if st != _b.FA_OK:
        raise _b.FaError(st, f"device error (site 0x{site:x})")
