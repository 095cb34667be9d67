// C ABI entry points: argument validation, workspace sizing, device error word,
// variant choice, and dispatch to the kernel launchers.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "fa.h"
#include "host.h"

namespace fa {
namespace {

thread_local int g_last_cuda_error = 0;
std::mutex g_mutex;
constexpr int kMaxDevices = 64;
int* g_err_word[kMaxDevices] = {};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_d(int d) { return padded_head_dim(d) != 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

fa_status validate_common(int B, int H, int N, int d, float scale, int causal) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!supported_d(d)) return FA_ERR_UNSUPPORTED;
  // B*H and B*H*N*d must fit the 32-bit grid/coordinate ranges the kernels use.
  const long long bh = (long long)B * H;
  if (bh > 0x7fffffffLL || (long long)N > 0x7fffffffLL / 2) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

}  // namespace

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_err_word[dev]) {
    int* w = nullptr;
    if (cudaMalloc(&w, 2 * sizeof(int)) != cudaSuccess) return nullptr;
    if (cudaMemset(w, 0, 2 * sizeof(int)) != cudaSuccess) {
      cudaFree(w);
      return nullptr;
    }
    g_err_word[dev] = w;
  }
  return g_err_word[dev];
}

int sm_count_cached() {
  static int sms[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    sms[dev] = n;
  }
  return sms[dev];
}

int head_group(int tiles_per_head, int BH) {
  const int t = tiles_per_head > 0 ? tiles_per_head : 1;
  const int g = (2 * sm_count_cached() + t - 1) / t;
  return g < 1 ? 1 : (g > BH ? BH : g);
}

int l2_head_group(double head_bytes, int BH, int tiles_per_head) {
  // About 96 MiB of re-read operands in flight stays well inside L2 next to the
  // other traffic.  A group keeps at least three waves of work items, so that
  // balancing heaviest-first inside it still has room (measured: fewer items per
  // group lost more to the imbalance than L2 reuse gained).
  const double per_head = head_bytes;
  double g = per_head > 0 ? (96.0 * 1024 * 1024) / per_head : (double)BH;
  const int t = tiles_per_head > 0 ? tiles_per_head : 1;
  g = std::max(g, std::ceil(3.0 * sm_count_cached() / t));
  const int gi = g < 1.0 ? 1 : (g > (double)BH ? BH : (int)g);
  // Equal-sized groups of at least gi heads: a small last group would start its
  // heaviest items last.
  const int ngroups = std::max(1, BH / gi);
  return (BH + ngroups - 1) / ngroups;
}

fa_status record_cuda_error(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return FA_ERR_LAUNCH;
}

fa_status make_tile_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                        int elem_bytes, int inner, int N, int BH, int box_inner, int box_rows,
                        CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return record_cuda_error(cudaErrorNotSupported);
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)inner * elem_bytes, (cuuint64_t)N * inner * elem_bytes};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return record_cuda_error(cudaErrorInvalidValue);
  return FA_OK;
}

// ------------------------------------------------------------------ profiling
namespace {
struct ProfRecord {
  int kind;
  cudaEvent_t a, b;
};
std::mutex g_prof_mutex;
bool g_prof_on = false;
std::vector<ProfRecord> g_prof;       // records of the current session
std::vector<cudaEvent_t> g_evt_pool;  // events reused across sessions
size_t g_prof_used_events = 0;
thread_local cudaEvent_t g_pending = nullptr;

cudaEvent_t pool_event() {
  if (g_prof_used_events < g_evt_pool.size()) return g_evt_pool[g_prof_used_events++];
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  g_evt_pool.push_back(e);
  ++g_prof_used_events;
  return e;
}
}  // namespace

void prof_before(int kind, cudaStream_t st) {
  (void)kind;
  std::lock_guard<std::mutex> lock(g_prof_mutex);
  if (!g_prof_on) return;
  g_pending = pool_event();
  if (g_pending) cudaEventRecord(g_pending, st);
}

void prof_after(int kind, cudaStream_t st) {
  std::lock_guard<std::mutex> lock(g_prof_mutex);
  if (!g_prof_on || !g_pending) return;
  cudaEvent_t b = pool_event();
  if (!b) return;
  cudaEventRecord(b, st);
  g_prof.push_back({kind, g_pending, b});
  g_pending = nullptr;
}

}  // namespace fa

using namespace fa;

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, void* stream) {
  fa_status s = validate_common(B, H, N, d, scale, causal);
  if (s != FA_OK) return s;
  if ((long long)B * H * N == 0) return FA_OK;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  return run_fwd(q, k, v, o, lse, B * H, N, d, scale, causal, 1, nullptr, (cudaStream_t)stream);
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int splits) {
  if (B < 0 || H < 0 || N < 0 || !supported_d(d)) return 0;
  if (splits < 1 || splits > FA_FWD_MAX_SPLITS) return 0;
  return splitkv_workspace_bytes(B * H, N, d, splits);
}

int fa_fwd_choose_splits(int B, int H, int N, int d, int causal) {
  if (validate_common(B, H, N, d, 1.f, causal) != FA_OK || (long long)B * H * N == 0) return 1;
  return choose_splits(B * H, N, d, causal);
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                         int N, int d, float scale, int causal, int splits, void* workspace,
                         size_t workspace_bytes, void* stream) {
  fa_status s = validate_common(B, H, N, d, scale, causal);
  if (s != FA_OK) return s;
  if (splits < 1 || splits > FA_FWD_MAX_SPLITS) return FA_ERR_INVALID_ARG;
  if ((long long)B * H * N == 0) return FA_OK;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  if (splits > 1 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                     workspace_bytes < splitkv_workspace_bytes(B * H, N, d, splits)))
    return FA_ERR_WORKSPACE;
  return run_fwd(q, k, v, o, lse, B * H, N, d, scale, causal, splits, workspace, (cudaStream_t)stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d, int variant) {
  if (B < 0 || H < 0 || N < 0 || !supported_d(d)) return 0;
  if (variant != FA_BWD_AUTO && variant != FA_BWD_5GEMM && variant != FA_BWD_7GEMM) return 0;
  const size_t bh = (size_t)B * H;
  const size_t npad = round_up((size_t)N, 128);
  size_t rows = 2 * round_up(4 * bh * npad, 256);  // log2-domain LSE and D per padded row
  // The variant's own needs: the 5-GEMM fp32 dQ accumulator (padded head dim) and
  // the partial dK / dV of the dK/dV kernel's query-range split.
  size_t five = 0, seven = 0;
  if (bwd_supported(d, FA_BWD_5GEMM))
    five = 4 * bh * npad * (size_t)padded_head_dim(d) + bwd_split_bytes(B * H, N, d, 1, FA_BWD_5GEMM);
  seven = bwd_split_bytes(B * H, N, d, 1, FA_BWD_7GEMM);
  // The split count depends on the mask; size for the larger of the two.
  if (bwd_supported(d, FA_BWD_5GEMM))
    five = std::max(five, 4 * bh * npad * (size_t)padded_head_dim(d) + bwd_split_bytes(B * H, N, d, 0, FA_BWD_5GEMM));
  seven = std::max(seven, bwd_split_bytes(B * H, N, d, 0, FA_BWD_7GEMM));
  const size_t extra = variant == FA_BWD_5GEMM ? five : variant == FA_BWD_7GEMM ? seven : std::max(five, seven);
  return rows + extra + 256;
}

// Measured on GB300 (bench.py --variant-table: 306 shapes, d = 64, 96 and 128,
// both masks, 1 to 512 heads, N = 512 to 16384, each form with its own
// few-heads splits; three runs): the 5-GEMM form was faster at 305, 305 and 299
// of 306 points, with the 7-GEMM form taking up to 2.6x its time (median 1.3x).
// The exceptions differed between the runs; those of the third (up to 23 %
// ahead, without the mask at 32 or 64 key tiles) were runs of the 5-GEMM form's
// slow mode at those shapes, and timed again the 5-GEMM form was ahead at each.
// So AUTO takes the 5-GEMM form wherever it exists (d <= 128); d = 192, 256 and
// 384 have only the 7-GEMM form.
int fa_bwd_choose(int B, int H, int N, int d, int causal) {
  (void)B;
  (void)H;
  (void)N;
  (void)causal;
  if (!bwd_supported(d, FA_BWD_5GEMM)) return FA_BWD_7GEMM;
  return FA_BWD_5GEMM;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, int variant, void* workspace, size_t workspace_bytes,
                 void* stream) {
  fa_status s = validate_common(B, H, N, d, scale, causal);
  if (s != FA_OK) return s;
  if (variant != FA_BWD_AUTO && variant != FA_BWD_5GEMM && variant != FA_BWD_7GEMM)
    return FA_ERR_INVALID_ARG;
  if ((long long)B * H * N == 0) return FA_OK;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  const int chosen = variant == FA_BWD_AUTO ? fa_bwd_choose(B, H, N, d, causal) : variant;
  if (!bwd_supported(d, chosen)) return FA_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < fa_bwd_workspace_size(B, H, N, d, chosen))
    return FA_ERR_WORKSPACE;
  return run_bwd(q, k, v, o, dO, lse, dq, dk, dv, B * H, N, d, scale, causal, chosen, workspace,
                 (cudaStream_t)stream);
}

int fa_bwd_query_parts(int B, int H, int N, int d, int causal, int variant) {
  if (validate_common(B, H, N, d, 1.f, causal) != FA_OK || (long long)B * H * N == 0) return 1;
  const int v = variant == FA_BWD_AUTO ? fa_bwd_choose(B, H, N, d, causal) : variant;
  if (!bwd_supported(d, v)) return 1;
  return choose_qsplit(B * H, N, d, causal, v);
}

int fa_bwd_force_query_parts(int parts) {
  if (parts < 0 || parts > FA_BWD_MAX_QUERY_PARTS) return FA_ERR_INVALID_ARG;
  force_qsplit(parts);
  return FA_OK;
}

int fa_bwd_key_parts(int B, int H, int N, int d, int causal, int variant) {
  if (validate_common(B, H, N, d, 1.f, causal) != FA_OK || (long long)B * H * N == 0) return 1;
  const int v = variant == FA_BWD_AUTO ? fa_bwd_choose(B, H, N, d, causal) : variant;
  if (!bwd_supported(d, v)) return 1;
  return choose_ksplit(B * H, N, d, causal, v);
}

int fa_bwd_force_key_parts(int parts) {
  if (parts < 0 || parts > FA_BWD_MAX_KEY_PARTS) return FA_ERR_INVALID_ARG;
  force_ksplit(parts);
  return FA_OK;
}

fa_status fa_get_device_error(void* stream, int* site) {
  if (site) *site = 0;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return record_cuda_error(e);
  int* w = device_error_word();
  if (!w) return record_cuda_error(cudaErrorMemoryAllocation);
  int h[2] = {0, 0};
  e = cudaMemcpy(h, w, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return record_cuda_error(e);
  if (h[0] != 0) {
    if (site) *site = h[1];
    cudaMemset(w, 0, sizeof(h));
    return FA_ERR_DEVICE_TIMEOUT;
  }
  return FA_OK;
}

int fa_last_cuda_error(void) { return g_last_cuda_error; }

const char* fa_strerror(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension or variant";
    case FA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case FA_ERR_LAUNCH: return "CUDA launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "in-kernel wait timed out";
  }
  return "unknown status";
}

int fa_profile_start(void) {
  std::lock_guard<std::mutex> lock(g_prof_mutex);
  g_prof.clear();
  g_prof_used_events = 0;
  g_prof_on = true;
  return FA_OK;
}

int fa_profile_stop(fa_profile* out) {
  std::lock_guard<std::mutex> lock(g_prof_mutex);
  g_prof_on = false;
  if (out) {
    for (int k = 0; k < FA_KERNEL_KINDS; ++k) {
      out->launches[k] = 0;
      out->ms[k] = 0.0;
    }
  }
  int status = FA_OK;
  for (const ProfRecord& r : g_prof) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      status = FA_ERR_LAUNCH;
      continue;
    }
    if (out && r.kind >= 0 && r.kind < FA_KERNEL_KINDS) {
      out->launches[r.kind] += 1;
      out->ms[r.kind] += ms;
    }
  }
  g_prof.clear();
  g_prof_used_events = 0;
  return status;
}

const char* fa_kernel_name(int kind) {
  switch (kind) {
    case FA_KERNEL_FWD: return "fwd";
    case FA_KERNEL_BWD_PRE: return "bwd_pre";
    case FA_KERNEL_BWD_KV5: return "bwd_kv5";
    case FA_KERNEL_BWD_CONV: return "bwd_conv";
    case FA_KERNEL_BWD_KV7: return "bwd_kv7";
    case FA_KERNEL_BWD_Q7: return "bwd_q7";
    case FA_KERNEL_FWD_MERGE: return "fwd_merge";
    case FA_KERNEL_BWD_KVSUM: return "bwd_kvsum";
    case FA_KERNEL_BWD_QSUM: return "bwd_qsum";
  }
  return "unknown";
}

int fa_fwd_launches(int B, int H, int N, int d) {
  if ((long long)B * H * N <= 0 || !supported_d(d)) return 0;
  return fwd_launch_count(d);
}

int fa_fwd_splitkv_launches(int B, int H, int N, int d, int splits) {
  if ((long long)B * H * N <= 0 || !supported_d(d) || splits < 1 || splits > FA_FWD_MAX_SPLITS) return 0;
  return fwd_launch_count(d) + (splits > 1 ? 1 : 0);
}

int fa_bwd_launches(int B, int H, int N, int d, int variant, int causal) {
  if ((long long)B * H * N <= 0 || !supported_d(d)) return 0;
  const int v = variant == FA_BWD_AUTO ? fa_bwd_choose(B, H, N, d, causal) : variant;
  if (!bwd_supported(d, v)) return 0;
  return bwd_launch_count(B * H, N, d, causal, v);
}

}  // extern "C"
