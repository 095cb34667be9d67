"""Torch-tensor convenience wrappers over the C ABI (marshalling only).

PyTorch supplies device memory and the current stream; the computation runs in
the CUDA library through ``binding``.  Tensors must be CUDA, bf16 (LSE fp32),
C-contiguous and shaped [B, H, N, d].
"""

from __future__ import annotations

import math

from . import binding as _b


def _validate(specs, device=None):
    """Rejects any operand that is not a contiguous CUDA tensor of its dtype and
    shape on one device, before a pointer of it can reach the library.  specs:
    (tensor, name, dtype, shape or None); dtypes and shapes are checked first."""
    import torch
    for t, name, dtype, shape in specs:
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch tensor")
        if t.dtype != dtype:
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor, not {t.dtype}")
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, not {tuple(t.shape)}")
    for t, name, dtype, _ in specs:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
        dev = device if device is not None else specs[0][0].device
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other operands on {dev}")


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
    if not isinstance(q, torch.Tensor) or q.dim() != 4:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    specs = [(q, "q", torch.bfloat16, None), (k, "k", torch.bfloat16, q.shape), (v, "v", torch.bfloat16, q.shape)]
    if out is not None:
        specs.append((out, "out", torch.bfloat16, q.shape))
    if lse is not None:
        specs.append((lse, "lse", torch.float32, (B, H, N)))
    _validate(specs)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if splits is None:
        splits = _b.fa_fwd_choose_splits(B, H, N, d, int(causal))
    if splits == 1:
        st = _b.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                       B, H, N, d, scale, int(causal), _stream(stream))
        if st != _b.FA_OK:
            raise _b.FaError(st, "fa_fwd")
        return o, l
    need = _b.fa_fwd_splitkv_workspace_size(B, H, N, d, splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    else:
        _validate([(workspace, "workspace", torch.uint8, None)], q.device)
        if workspace.numel() < need:
            raise ValueError(f"workspace holds {workspace.numel()} bytes, {need} are needed")
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
    if not isinstance(q, torch.Tensor) or q.dim() != 4:
        raise ValueError("q, k, v, o, do must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    if grads is not None and len(grads) != 3:
        raise ValueError("grads must be (dq, dk, dv)")
    specs = [(q, "q", torch.bfloat16, None)] + [(t, n, torch.bfloat16, q.shape)
                                                for t, n in ((k, "k"), (v, "v"), (o, "o"), (do, "do"))]
    specs.append((lse, "lse", torch.float32, (B, H, N)))
    if grads is not None:
        specs += [(t, n, torch.bfloat16, q.shape) for t, n in zip(grads, ("dq", "dk", "dv"))]
    if workspace is not None:
        specs.append((workspace, "workspace", torch.uint8, None))
    _validate(specs)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    need = _b.fa_bwd_workspace_size(B, H, N, d, variant)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    elif workspace.numel() < need:
        raise ValueError(f"workspace holds {workspace.numel()} bytes, {need} are needed")
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
