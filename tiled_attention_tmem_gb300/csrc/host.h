// Host-side helpers shared by the launcher translation units (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// Device error word (two ints) of the current device, created on first use.
// Returns nullptr if it could not be created.
int* device_error_word();

// Records a CUDA runtime error code for fa_last_cuda_error and returns FA_ERR_LAUNCH.
fa_status record_cuda_error(cudaError_t e);

// Launches the watchdog self-test kernel (one warp whose bounded wait expires)
// against the given device error word (watchdog.cu).
fa_status launch_watchdog_selftest(int* err, cudaStream_t st);

// Builds a 3-D TMA descriptor over a contiguous [BH, N, inner] tensor:
// dims {inner, N, BH}, box {64, box_rows, 1}, 128-byte swizzle, zero fill out of bounds.
fa_status make_tile_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                        int elem_bytes, int inner, int N, int BH, int box_inner, int box_rows,
                        CUtensorMapSwizzle swizzle);

// Heads per launch-order group: enough heads for about two waves of blocks on
// this device (at least 1, at most BH).  The statically scheduled kernels use
// one group of all heads under the causal mask, where heaviest-tile-first
// across every head balances better than locality helps.
int head_group(int tiles_per_head, int BH);
// Heads per launch-order group so that the operands each head keeps re-reading
// (head_bytes per head: K and V for the forward; Q, K, V, dO and the fp32 dQ
// accumulator for the backward) fit in L2, with at least three waves of work
// items per group so that heaviest-first ordering inside a group still balances.
int l2_head_group(double head_bytes, int BH, int tiles_per_head);

// Multiprocessor count of the current device (cached per device).
int sm_count_cached();

// Profiling markers (no-ops unless fa_profile_start is active).
void prof_before(int kind, cudaStream_t st);
void prof_after(int kind, cudaStream_t st);

// Kernel launch helper: sets the dynamic shared memory limit and launches with
// programmatic stream serialization, so the kernel can be scheduled while the
// previous kernel in the stream finishes (every kernel of this library waits
// for it with griddepcontrol.wait before touching memory).
template <class Kernel, class Params>
fa_status launch(int kind, Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                 const Params& p) {
  cudaError_t e = cudaSuccess;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return record_cuda_error(e);
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before(kind, st);
  e = cudaLaunchKernelEx(&cfg, kernel, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  prof_after(kind, st);
  if (e != cudaSuccess) return record_cuda_error(e);
  return FA_OK;
}

// Forward launcher (fwd.cu).  Arguments already validated.  splits > 1 runs the
// split-KV form: `workspace` (splitkv_workspace_bytes, 256-byte aligned) holds
// the fp32 parts at offset 0 and their log-sum-exps at splitkv_lse_offset.
fa_status run_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int N,
                  int d, float scale, int causal, int splits, void* workspace, cudaStream_t st);
constexpr int kMaxSplits = 16;
size_t splitkv_lse_offset(int BH, int N, int d, int splits);
size_t splitkv_workspace_bytes(int BH, int N, int d, int splits);
// Parts per query block that the split-KV cost model predicts fastest (1: no split).
int choose_splits(int BH, int N, int d, int causal);
int fwd_launch_count(int d);

// Head dims the kernels support and the head dim (64, 128, 256 or 384) whose
// workspace layout, preprocess and variant rules serve each: 96 runs the 128
// kernels on zero-padded tiles; 192 has its own forward, dK/dV and dQ kernels
// but the 256 preprocess and rules (no 5-GEMM); 384 has its own kernels and
// the 7-GEMM form only.  0 if unsupported.
inline int padded_head_dim(int d) {
  return d == 64 ? 64 : (d == 96 || d == 128) ? 128 : (d == 192 || d == 256) ? 256 : d == 384 ? 384 : 0;
}

// Backward launchers (bwd.cu).  Arguments already validated; workspace sized.
fa_status run_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                  const float* lse, void* dq, void* dk, void* dv, int BH, int N, int d,
                  float scale, int causal, int variant, void* workspace, cudaStream_t st);
bool bwd_supported(int d, int variant);
int bwd_launch_count(int BH, int N, int d, int causal, int variant);
// Query parts per key tile of the dK/dV kernel (1: no split) and the workspace
// bytes of the fp32 partials of both splits (0 without a split).
int choose_qsplit(int BH, int N, int d, int causal, int variant);
// Benchmark hook behind fa_bwd_force_query_parts (0: the automatic choice).
void force_qsplit(int parts);
// Key parts per query tile of the 7-GEMM dQ kernel (1: no split; always 1 for the
// 5-GEMM form) and its benchmark hook behind fa_bwd_force_key_parts.
int choose_ksplit(int BH, int N, int d, int causal, int variant);
void force_ksplit(int parts);
size_t bwd_split_bytes(int BH, int N, int d, int causal, int variant);

}  // namespace fa
