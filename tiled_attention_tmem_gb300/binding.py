"""ctypes binding of the C ABI in ``include/fa.h`` (argument marshalling only).

The functions here carry the C names and take raw device pointers (ints),
sizes and a CUDA stream handle; every step of the computation runs in the
CUDA library.  If ``libfa_gb300.so`` has not been built this module raises on
first use: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa_gb300.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_WORKSPACE = 4
FA_ERR_LAUNCH = 5
FA_ERR_DEVICE_TIMEOUT = 6

FA_FWD_MAX_SPLITS = 64

FA_BWD_AUTO = 0
FA_BWD_5GEMM = 5
FA_BWD_7GEMM = 7

# Every symbol the header declares, with its ctypes signature.
_VP = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
SIGNATURES = {
    "fa_fwd": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _F, _I, _VP]),
    "fa_fwd_splitkv_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "fa_fwd_splitkv": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _F, _I, _I, _VP, _SZ, _VP]),
    "fa_fwd_choose_splits": (_I, [_I, _I, _I, _I, _I]),
    "fa_bwd_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "fa_bwd": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                    _I, _I, _I, _I, _F, _I, _I, _VP, _SZ, _VP]),
    "fa_bwd_noalloc": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                            _I, _I, _I, _I, _F, _I, _I, _VP]),
    "fa_bwd_noalloc_device_error": (_I, [_VP, ctypes.POINTER(_I)]),
    "fa_bwd_noalloc_watchdog_selftest": (_I, [_VP]),
    "fa_bwd_query_parts": (_I, [_I, _I, _I, _I, _I, _I]),
    "fa_bwd_force_query_parts": (_I, [_I]),
    "fa_bwd_key_parts": (_I, [_I, _I, _I, _I, _I, _I]),
    "fa_bwd_force_key_parts": (_I, [_I]),
    "fa_bwd_choose": (_I, [_I, _I, _I, _I, _I]),
    "fa_get_device_error": (_I, [_VP, ctypes.POINTER(_I)]),
    "fa_watchdog_selftest": (_I, [_VP]),
    "fa_last_cuda_error": (_I, []),
    "fa_strerror": (ctypes.c_char_p, [_I]),
    "fa_profile_start": (_I, []),
    "fa_profile_stop": (_I, [_VP]),
    "fa_kernel_name": (ctypes.c_char_p, [_I]),
    "fa_ex2_probe": (_I, [_VP, _I, _I, ctypes.POINTER(ctypes.c_longlong), _VP]),
    "fa_fwd_launches": (_I, [_I, _I, _I, _I]),
    "fa_fwd_splitkv_launches": (_I, [_I, _I, _I, _I, _I]),
    "fa_bwd_launches": (_I, [_I, _I, _I, _I, _I, _I]),
}

_lib = None
_lock = threading.Lock()


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa_strerror(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """Loads the shared library once; raises if it is missing."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with tiled_attention_tmem_gb300.build "
                        "(or __graft_entry__.build()); there is no CPU fallback")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def fa_strerror(status: int) -> str:
    return lib().fa_strerror(status).decode()


def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> int:
    return lib().fa_fwd(q, k, v, o, lse, B, H, N, d, float(scale), int(causal), stream)


def fa_fwd_splitkv_workspace_size(B, H, N, d, splits) -> int:
    return lib().fa_fwd_splitkv_workspace_size(B, H, N, d, splits)


def fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, splits, workspace, workspace_bytes,
                   stream) -> int:
    return lib().fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, float(scale), int(causal), int(splits),
                                workspace, workspace_bytes, stream)


def fa_fwd_choose_splits(B, H, N, d, causal) -> int:
    return lib().fa_fwd_choose_splits(B, H, N, d, int(causal))


def fa_bwd_workspace_size(B, H, N, d, variant) -> int:
    return lib().fa_bwd_workspace_size(B, H, N, d, variant)


def fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, variant,
           workspace, workspace_bytes, stream) -> int:
    return lib().fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, float(scale), int(causal),
                        variant, workspace, workspace_bytes, stream)


def fa_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, variant, stream) -> int:
    """The backward without a workspace: scratch lives in the library's static device array."""
    return lib().fa_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, float(scale), int(causal),
                                variant, stream)


FA_NOALLOC_SCRATCH_BYTES = 64 << 20


def fa_bwd_noalloc_device_error(stream) -> tuple[int, int]:
    """(status, site) of the no-alloc backward's own error word; reading clears it."""
    site = _I(0)
    status = lib().fa_bwd_noalloc_device_error(stream, ctypes.byref(site))
    return status, site.value


def fa_bwd_noalloc_watchdog_selftest(stream) -> int:
    return lib().fa_bwd_noalloc_watchdog_selftest(stream)


def fa_bwd_query_parts(B, H, N, d, causal, variant) -> int:
    return lib().fa_bwd_query_parts(B, H, N, d, int(causal), variant)


def fa_bwd_force_query_parts(parts) -> int:
    return lib().fa_bwd_force_query_parts(int(parts))


def fa_bwd_key_parts(B, H, N, d, causal, variant) -> int:
    return lib().fa_bwd_key_parts(B, H, N, d, int(causal), variant)


def fa_bwd_force_key_parts(parts) -> int:
    return lib().fa_bwd_force_key_parts(int(parts))


def fa_bwd_choose(B, H, N, d, causal) -> int:
    return lib().fa_bwd_choose(B, H, N, d, int(causal))


def fa_get_device_error(stream) -> tuple[int, int]:
    site = _I(0)
    status = lib().fa_get_device_error(stream, ctypes.byref(site))
    return status, site.value


def fa_watchdog_selftest(stream) -> int:
    return lib().fa_watchdog_selftest(stream)


def fa_last_cuda_error() -> int:
    return lib().fa_last_cuda_error()


def fa_ex2_probe(sink, blocks, iters, stream) -> tuple[int, int]:
    """Launches the exponential-unit probe; returns (status, ex2 evaluations launched)."""
    count = ctypes.c_longlong(0)
    status = lib().fa_ex2_probe(sink, blocks, iters, ctypes.byref(count), stream)
    return status, count.value


def fa_fwd_launches(B, H, N, d) -> int:
    return lib().fa_fwd_launches(B, H, N, d)


def fa_fwd_splitkv_launches(B, H, N, d, splits) -> int:
    return lib().fa_fwd_splitkv_launches(B, H, N, d, splits)


def fa_bwd_launches(B, H, N, d, variant, causal=0) -> int:
    return lib().fa_bwd_launches(B, H, N, d, variant, int(causal))


FA_KERNEL_KINDS = 9


class FaProfile(ctypes.Structure):
    _fields_ = [("launches", _I * FA_KERNEL_KINDS), ("ms", ctypes.c_double * FA_KERNEL_KINDS)]


def fa_profile_start() -> int:
    return lib().fa_profile_start()


def fa_profile_stop() -> dict:
    """Returns {kernel name: (launches, total ms)} for the kernels launched since start."""
    prof = FaProfile()
    st = lib().fa_profile_stop(ctypes.byref(prof))
    if st != FA_OK:
        raise FaError(st, "fa_profile_stop")
    return {lib().fa_kernel_name(k).decode(): (prof.launches[k], prof.ms[k])
            for k in range(FA_KERNEL_KINDS)}
