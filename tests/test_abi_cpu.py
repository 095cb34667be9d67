"""The C-ABI library loads, exports every declared symbol, and validates arguments.

These tests need no GPU: every call below is rejected (or is a no-op) before
any CUDA work is issued.
"""

import ctypes
import os
import re
import shutil
import subprocess

import pytest

from tiled_attention_tmem_gb300 import binding as b
from tiled_attention_tmem_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return b.lib()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "fa_fwd" in names and "fa_bwd" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in b.SIGNATURES, f"binding lacks {n}"


A = 1 << 20  # a 16-byte aligned fake address; never dereferenced


def test_fwd_validation(lib):
    ok = dict(B=1, H=2, N=128, d=64, scale=0.125, causal=0)

    def call(q=A, k=A, v=A, o=A, lse=A, **kw):
        a = {**ok, **kw}
        return b.fa_fwd(q, k, v, o, lse, a["B"], a["H"], a["N"], a["d"], a["scale"], a["causal"], None)

    assert call(d=80) == b.FA_ERR_UNSUPPORTED
    assert call(d=160) == b.FA_ERR_UNSUPPORTED
    assert call(d=32) == b.FA_ERR_UNSUPPORTED
    assert call(N=-1) == b.FA_ERR_INVALID_ARG
    assert call(scale=0.0) == b.FA_ERR_INVALID_ARG
    assert call(scale=-0.5) == b.FA_ERR_INVALID_ARG
    assert call(scale=float("nan")) == b.FA_ERR_INVALID_ARG
    assert call(scale=float("inf")) == b.FA_ERR_INVALID_ARG
    assert call(causal=2) == b.FA_ERR_INVALID_ARG
    assert call(q=0) == b.FA_ERR_INVALID_ARG
    assert call(lse=0) == b.FA_ERR_INVALID_ARG
    assert call(k=A + 8) == b.FA_ERR_MISALIGNED
    assert call(lse=A + 4) == b.FA_ERR_MISALIGNED
    # Empty problems are a no-op and never touch the (null) pointers.
    assert call(q=0, k=0, v=0, o=0, lse=0, N=0) == b.FA_OK
    assert call(q=0, k=0, v=0, o=0, lse=0, B=0) == b.FA_OK


def test_bwd_validation(lib):
    ws = b.fa_bwd_workspace_size(1, 2, 128, 64, b.FA_BWD_AUTO)
    assert ws > 0

    def call(variant=b.FA_BWD_7GEMM, workspace=A, wsb=ws, d=64, scale=0.125, dq=A, lse=A):
        return b.fa_bwd(A, A, A, A, A, lse, dq, A, A, 1, 2, 128, d, scale, 0, variant,
                        workspace, wsb, None)

    assert call(variant=3) == b.FA_ERR_INVALID_ARG
    assert call(d=80) == b.FA_ERR_UNSUPPORTED
    assert call(scale=0.0) == b.FA_ERR_INVALID_ARG
    assert call(dq=0) == b.FA_ERR_INVALID_ARG
    assert call(dq=A + 2) == b.FA_ERR_MISALIGNED
    if b.lib().fa_bwd_launches(1, 2, 128, 64, b.FA_BWD_7GEMM, 0) > 0:
        assert call(workspace=0) == b.FA_ERR_WORKSPACE
        assert call(workspace=A + 16) == b.FA_ERR_WORKSPACE
        ws7 = b.fa_bwd_workspace_size(1, 2, 128, 64, b.FA_BWD_7GEMM)
        assert call(wsb=ws7 - 16) == b.FA_ERR_WORKSPACE
        ws5 = b.fa_bwd_workspace_size(1, 2, 128, 64, b.FA_BWD_5GEMM)
        assert call(variant=b.FA_BWD_5GEMM, wsb=ws5 - 16) == b.FA_ERR_WORKSPACE
        # head dim 256 has no 5-GEMM kernel
        assert b.fa_bwd(A, A, A, A, A, A, A, A, A, 1, 2, 128, 256, 0.0625, 0, b.FA_BWD_5GEMM,
                        A, ws5, None) == b.FA_ERR_UNSUPPORTED


def test_workspace_sizes(lib):
    for d in (64, 96, 128, 192, 256):
        w7 = b.fa_bwd_workspace_size(2, 3, 300, d, b.FA_BWD_7GEMM)
        assert w7 >= 4 * 6 * 384
        wa = b.fa_bwd_workspace_size(2, 3, 300, d, b.FA_BWD_AUTO)
        assert wa >= w7
        if b.lib().fa_bwd_launches(2, 3, 300, d, b.FA_BWD_5GEMM, 0) > 0:
            w5 = b.fa_bwd_workspace_size(2, 3, 300, d, b.FA_BWD_5GEMM)
            assert w5 >= 4 * 6 * 384 * (d + 1)
    # head dim 96 runs on zero-padded 128 tiles: the fp32 dQ accumulator has the
    # padded width.  Head dim 192 has no 5-GEMM kernel (its dV, dK and dQ
    # accumulators do not fit TMEM together).
    assert (b.fa_bwd_workspace_size(2, 3, 300, 96, b.FA_BWD_5GEMM)
            == b.fa_bwd_workspace_size(2, 3, 300, 128, b.FA_BWD_5GEMM))
    assert b.fa_bwd_workspace_size(2, 3, 300, 192, b.FA_BWD_5GEMM) == 0 or \
        b.lib().fa_bwd_launches(2, 3, 300, 192, b.FA_BWD_5GEMM, 0) == 0
    assert b.fa_bwd_choose(1, 1, 128, 192, 0) == b.FA_BWD_7GEMM
    assert b.fa_bwd_workspace_size(1, 1, 128, 100, b.FA_BWD_AUTO) == 0
    assert b.fa_bwd_workspace_size(1, 1, 128, 64, 9) == 0


def test_splitkv_validation(lib):
    """Argument checks of the split-KV forward (none of these launch anything)."""
    def call(B=1, H=2, N=128, d=64, scale=0.125, causal=0, splits=2, ws=A, wsb=1 << 30, q=A, lse=A):
        return b.fa_fwd_splitkv(q, A, A, A, lse, B, H, N, d, scale, causal, splits, ws, wsb, None)

    assert call(d=80) == b.FA_ERR_UNSUPPORTED
    assert call(splits=0) == b.FA_ERR_INVALID_ARG
    assert call(splits=-3) == b.FA_ERR_INVALID_ARG
    assert call(splits=b.FA_FWD_MAX_SPLITS + 1) == b.FA_ERR_INVALID_ARG
    assert call(scale=float("nan")) == b.FA_ERR_INVALID_ARG
    assert call(q=0) == b.FA_ERR_INVALID_ARG
    assert call(lse=A + 4) == b.FA_ERR_MISALIGNED
    assert call(ws=0) == b.FA_ERR_WORKSPACE
    assert call(ws=A + 16) == b.FA_ERR_WORKSPACE  # 16- but not 256-byte aligned
    need = b.fa_fwd_splitkv_workspace_size(1, 2, 128, 64, 2)
    assert call(wsb=need - 1) == b.FA_ERR_WORKSPACE
    assert call(q=0, lse=0, ws=0, N=0) == b.FA_OK


def test_splitkv_workspace_and_launches(lib):
    def r256(x):
        return (x + 255) // 256 * 256
    for d in (64, 96, 128, 192, 256):
        for s in (2, 3, 16, b.FA_FWD_MAX_SPLITS):
            got = b.fa_fwd_splitkv_workspace_size(2, 3, 300, d, s)
            assert got == r256(4 * s * 6 * 300 * d) + r256(4 * s * 6 * 300), (d, s)
        assert b.fa_fwd_splitkv_workspace_size(2, 3, 300, d, 1) == 0
        assert b.fa_fwd_splitkv_launches(2, 3, 300, d, 1) == 1
        assert b.fa_fwd_splitkv_launches(2, 3, 300, d, 5) == 2
    assert b.fa_fwd_splitkv_workspace_size(2, 3, 300, 64, 0) == 0
    assert b.fa_fwd_splitkv_workspace_size(2, 3, 300, 64, b.FA_FWD_MAX_SPLITS + 1) == 0
    assert b.fa_fwd_splitkv_workspace_size(2, 3, 300, 100, 2) == 0
    assert b.fa_fwd_splitkv_launches(2, 3, 0, 64, 2) == 0
    assert b.fa_fwd_splitkv_launches(2, 3, 300, 64, 0) == 0


def test_split_choice(lib):
    """The split-KV cost model: no split once the query blocks fill the SMs, a split
    for one long head (8192 rows: 32 or 64 query blocks), never more than 16 parts,
    at least two key tiles per part, 1 for invalid shapes."""
    assert b.fa_fwd_choose_splits(4, 16, 2048, 128, 1) == 1
    assert b.fa_fwd_choose_splits(16, 16, 512, 64, 0) == 1
    for d in (64, 96, 128, 192, 256):
        for causal in (0, 1):
            s = b.fa_fwd_choose_splits(1, 1, 8192, d, causal)
            assert 2 <= s <= 16, (d, causal, s)
            for N in (1, 100, 1000, 5000, 70000):
                s = b.fa_fwd_choose_splits(1, 2, N, d, causal)
                assert 1 <= s <= 16
                tiles = -(-N // (128 if d <= 128 else 64))
                assert s == 1 or tiles // s >= 2
    assert b.fa_fwd_choose_splits(1, 1, 128, 100, 0) == 1
    assert b.fa_fwd_choose_splits(1, 1, 0, 128, 0) == 1


def test_strerror(lib):
    for s in range(7):
        assert b.fa_strerror(s)
    assert b.fa_strerror(99) == "unknown status"


def test_launch_counts(lib):
    assert b.fa_fwd_launches(1, 1, 0, 64) == 0
    assert b.fa_fwd_launches(1, 1, 128, 64) == 1


def test_no_cpu_fallback_when_library_missing(tmp_path, monkeypatch):
    """The binding raises instead of computing anything when the .so is absent."""
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(b, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        b.fa_fwd(A, A, A, A, A, 1, 1, 128, 64, 0.125, 0, None)


def test_bwd_noalloc_validation(lib):
    """Argument checks of the allocation-free backward (none of these launch anything)."""
    def call(B=1, H=2, N=128, d=64, scale=0.125, causal=0, variant=b.FA_BWD_7GEMM, q=A, dq=A):
        return b.fa_bwd_noalloc(q, A, A, A, A, A, dq, A, A, B, H, N, d, scale, causal, variant, None)

    assert call(variant=3) == b.FA_ERR_INVALID_ARG
    assert call(scale=0.0) == b.FA_ERR_INVALID_ARG
    assert call(causal=2) == b.FA_ERR_INVALID_ARG
    assert call(B=-1) == b.FA_ERR_INVALID_ARG
    assert call(d=80) == b.FA_ERR_UNSUPPORTED
    assert call(d=160) == b.FA_ERR_UNSUPPORTED
    assert call(q=0) == b.FA_ERR_INVALID_ARG
    assert call(dq=A + 2) == b.FA_ERR_MISALIGNED
    assert call(N=0) == b.FA_OK  # empty problem: no-op
    # head dims above 128 have no 5-GEMM kernel
    assert call(d=256, variant=b.FA_BWD_5GEMM) == b.FA_ERR_UNSUPPORTED
    assert call(d=192, variant=b.FA_BWD_5GEMM) == b.FA_ERR_UNSUPPORTED
    assert call(d=384, variant=b.FA_BWD_5GEMM) == b.FA_ERR_UNSUPPORTED
    assert call(d=320) == b.FA_ERR_UNSUPPORTED
    # scratch beyond the static array is refused before anything is launched
    big = dict(B=64, H=64, N=8192)
    assert call(d=128, variant=b.FA_BWD_7GEMM, **big) == b.FA_ERR_WORKSPACE
    assert call(d=128, variant=b.FA_BWD_5GEMM, **big) == b.FA_ERR_WORKSPACE


C_CLIENT = r"""
#include <stdio.h>
#include <stddef.h>
#include "fa.h"

/* A C caller of the boundary: only calls that are rejected or answered before
   any CUDA work is issued. */
int main(void) {
  int fails = 0;
  fa_profile prof;
  if (fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 128, 80, 0.125f, 0, NULL) != FA_ERR_UNSUPPORTED) fails |= 1;
  if (fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 0, 64, 0.125f, 0, NULL) != FA_OK) fails |= 2;
  if (fa_fwd_splitkv(NULL, NULL, NULL, NULL, NULL, 1, 1, 128, 64, 0.125f, 0, 0, NULL, 0, NULL)
      != FA_ERR_INVALID_ARG) fails |= 4;
  if (fa_bwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 1, 128, 64, 0.125f, 0, 9, NULL, 0, NULL)
      != FA_ERR_INVALID_ARG) fails |= 8;
  if (fa_bwd_workspace_size(1, 1, 128, 100, FA_BWD_AUTO) != 0) fails |= 16;
  if (fa_fwd_splitkv_workspace_size(1, 1, 128, 64, 2) != (size_t)(4 * 2 * 128 * 64 + 4 * 2 * 128)) fails |= 32;
  if (fa_strerror(FA_ERR_WORKSPACE) == NULL || fa_kernel_name(FA_KERNEL_FWD_MERGE) == NULL) fails |= 64;
  if (fa_fwd_splitkv_launches(1, 1, 128, 64, 2) != 2 || fa_fwd_launches(1, 1, 128, 64) != 1) fails |= 128;
  if (sizeof(prof.launches) / sizeof(prof.launches[0]) != FA_KERNEL_KINDS) fails |= 256;
  printf("%d\n", fails);
  return fails != 0;
}
"""


def test_header_is_plain_c_and_a_c_program_links_the_library(lib, tmp_path):
    """include/fa.h compiles as strict C99, and a C program linked against the
    shared library gets the documented answers from calls that launch nothing."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(b.LIB_PATH)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        f"-I{os.path.join(ROOT, 'include')}", str(src), "-o", str(exe),
                        f"-L{libdir}", "-l:libfa_gb300.so", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == "0", out.stdout + out.stderr


def test_noalloc_source_calls_no_allocator():
    """The allocation-free backward's translation unit names no allocating call: no
    cudaMalloc / cudaFree family, and not the lazily cudaMalloc'ed error word of the
    workspace entry points."""
    src = open(os.path.join(ROOT, "tiled_attention_tmem_gb300", "csrc", "bwd_noalloc.cu")).read()
    code = re.sub(r"//[^\n]*", "", re.sub(r"/\*.*?\*/", "", src, flags=re.S))
    for banned in ("cudaMalloc", "cudaFree", "cuMemAlloc", "cuMemFree", "device_error_word", "malloc(",
                   "new ", "std::vector"):
        assert banned not in code, banned


def test_query_parts_override(lib):
    """The benchmark hook forces the dK/dV kernel's query-part count: launch count,
    workspace and the reported count follow it, and 0 restores the automatic rule."""
    B, H, N, d = 1, 64, 2048, 128  # many key tiles: the automatic rule does not split
    try:
        assert b.fa_bwd_query_parts(B, H, N, d, 1, b.FA_BWD_5GEMM) == 1
        base_ws = b.fa_bwd_workspace_size(B, H, N, d, b.FA_BWD_5GEMM)
        assert b.fa_bwd_launches(B, H, N, d, b.FA_BWD_5GEMM, 1) == 3
        assert b.fa_bwd_force_query_parts(3) == b.FA_OK
        assert b.fa_bwd_query_parts(B, H, N, d, 1, b.FA_BWD_5GEMM) == 3
        assert b.fa_bwd_launches(B, H, N, d, b.FA_BWD_5GEMM, 1) == 4
        # fp32 partial dK and dV for three parts
        assert b.fa_bwd_workspace_size(B, H, N, d, b.FA_BWD_5GEMM) == base_ws + 2 * 4 * 3 * B * H * N * d
        assert b.fa_bwd_force_query_parts(-1) == b.FA_ERR_INVALID_ARG
        assert b.fa_bwd_force_query_parts(17) == b.FA_ERR_INVALID_ARG
    finally:
        assert b.fa_bwd_force_query_parts(0) == b.FA_OK
    assert b.fa_bwd_query_parts(B, H, N, d, 1, b.FA_BWD_5GEMM) == 1
    assert b.fa_bwd_workspace_size(B, H, N, d, b.FA_BWD_5GEMM) == base_ws


def test_key_parts_override(lib):
    """The benchmark hook forces the dQ kernel's key-part count (7-GEMM only): launch
    count, workspace and the reported count follow it; the 5-GEMM form has no dQ
    kernel and stays at one part; 0 restores the automatic rule."""
    B, H, N, d = 1, 64, 2048, 128  # many query tiles: the automatic rule does not split
    try:
        assert b.fa_bwd_key_parts(B, H, N, d, 1, b.FA_BWD_7GEMM) == 1
        base7 = b.fa_bwd_workspace_size(B, H, N, d, b.FA_BWD_7GEMM)
        base5 = b.fa_bwd_workspace_size(B, H, N, d, b.FA_BWD_5GEMM)
        assert b.fa_bwd_launches(B, H, N, d, b.FA_BWD_7GEMM, 1) == 3
        assert b.fa_bwd_force_key_parts(5) == b.FA_OK
        assert b.fa_bwd_key_parts(B, H, N, d, 1, b.FA_BWD_7GEMM) == 5
        assert b.fa_bwd_key_parts(B, H, N, d, 1, b.FA_BWD_5GEMM) == 1
        assert b.fa_bwd_launches(B, H, N, d, b.FA_BWD_7GEMM, 1) == 4
        assert b.fa_bwd_launches(B, H, N, d, b.FA_BWD_5GEMM, 1) == 3
        # fp32 partial dQ for five parts; the 5-GEMM workspace is unchanged
        assert b.fa_bwd_workspace_size(B, H, N, d, b.FA_BWD_7GEMM) == base7 + 4 * 5 * B * H * N * d
        assert b.fa_bwd_workspace_size(B, H, N, d, b.FA_BWD_5GEMM) == base5
        # both splits at once: both partial sums and both summing kernels
        assert b.fa_bwd_force_query_parts(2) == b.FA_OK
        assert b.fa_bwd_launches(B, H, N, d, b.FA_BWD_7GEMM, 1) == 5
        assert b.fa_bwd_workspace_size(B, H, N, d, b.FA_BWD_7GEMM) == base7 + 4 * (5 + 2 * 2) * B * H * N * d
        assert b.fa_bwd_force_key_parts(-1) == b.FA_ERR_INVALID_ARG
        assert b.fa_bwd_force_key_parts(17) == b.FA_ERR_INVALID_ARG
    finally:
        assert b.fa_bwd_force_key_parts(0) == b.FA_OK
        assert b.fa_bwd_force_query_parts(0) == b.FA_OK
    assert b.fa_bwd_key_parts(B, H, N, d, 1, b.FA_BWD_7GEMM) == 1
    assert b.fa_bwd_workspace_size(B, H, N, d, b.FA_BWD_7GEMM) == base7


def test_key_split_for_few_heads(lib):
    """Few heads under the causal mask: the dQ kernel's query tiles are far fewer
    than the SMs, so the rule splits their key ranges (at most 8 parts, at least
    512 keys per part), and the workspace holds the partial sums for either mask."""
    assert b.fa_bwd_key_parts(1, 1, 4096, 256, 1, b.FA_BWD_7GEMM) == 8
    assert b.fa_bwd_key_parts(1, 1, 1024, 256, 1, b.FA_BWD_7GEMM) == 2
    assert b.fa_bwd_key_parts(1, 1, 4096, 128, 1, b.FA_BWD_AUTO) == 1  # AUTO: 5-GEMM, no dQ kernel
    for causal in (0, 1):
        k = b.fa_bwd_key_parts(1, 1, 4096, 256, causal, b.FA_BWD_7GEMM)
        qp = b.fa_bwd_query_parts(1, 1, 4096, 256, causal, b.FA_BWD_7GEMM)
        need = 2 * 4 * 4096 + 4 * k * 4096 * 256 + (2 * 4 * qp * 4096 * 256 if qp > 1 else 0)
        assert b.fa_bwd_workspace_size(1, 1, 4096, 256, b.FA_BWD_7GEMM) >= need
