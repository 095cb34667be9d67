// fa_bwd_noalloc: the backward with its scratch in a static device array.
//
// Who needs this: callers that cannot allocate device memory themselves, for
// example code running inside an allocator callback, a memory-capped plugin
// host, or a runtime that hands out only the input and output buffers.  fa_bwd
// needs a caller-provided workspace (and creates the library's device error
// word with cudaMalloc on first use), so such callers cannot use it.  This
// entry point allocates nothing: the fp32 row statistics, the fp32 dQ
// accumulator and the error word live in one file-scope __device__ array.
//
// The array costs kScratchBytes of device memory on every GPU that loads this
// library, held until the process exits.  Every call shares it, so calls that
// overlap on the GPU (different streams, or different host threads) race on it
// and must be serialised by the caller.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "bwd.cuh"
#include "host.h"

namespace fa {
namespace {

constexpr size_t kErrSlot = 256;                         // error word (2 ints) + padding
constexpr size_t kScratchBytes = FA_NOALLOC_SCRATCH_BYTES;  // workspace part
static __device__ __align__(256) unsigned char g_noalloc_scratch[kErrSlot + kScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_setup_mutex;
unsigned char* g_scratch_addr[kMaxDev] = {};

// Device address of the static array on the current device.  The host-side
// name g_noalloc_scratch is only a stand-in, never a device address.  Looked
// up once per device; returns nullptr if the runtime refuses.
unsigned char* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      record_cuda_error(e == cudaSuccess ? cudaErrorInvalidSymbol : e);
      return nullptr;
    }
    g_scratch_addr[dev] = static_cast<unsigned char*>(ptr);
  }
  return g_scratch_addr[dev];
}

size_t a256(size_t x) { return (x + 255) / 256 * 256; }

size_t scratch_need(int BH, int Npad, int d, bool five) {
  const size_t rows = (size_t)BH * Npad;
  return 2 * a256(4 * rows) + (five ? 4 * rows * (size_t)d : 0);
}

int sms() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

template <class KV, class Q7, int D>
fa_status run(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
              void* dq, void* dk, void* dv, int BH, int N, int hd, float scale, int causal, bool five,
              unsigned char* base, cudaStream_t st) {
  const int Npad = (N + 127) / 128 * 128;
  int* err = reinterpret_cast<int*>(base);
  int* sched = reinterpret_cast<int*>(base + 64);  // work-item counters, zeroed by the preprocess kernel
  unsigned char* ws = base + kErrSlot;
  float* lse2 = reinterpret_cast<float*>(ws);
  float* dd = reinterpret_cast<float*>(ws + a256(4 * (size_t)BH * Npad));
  float* dqacc = five ? reinterpret_cast<float*>(ws + 2 * a256(4 * (size_t)BH * Npad)) : nullptr;
  cudaError_t e = cudaMemsetAsync(err, 0, 2 * sizeof(int), st);
  if (e != cudaSuccess) return record_cuda_error(e);

  PreParams pp{static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dO), lse, lse2, dd, dqacc, N, Npad,
               BH, hd, sched};
  const long long pre_threads = (long long)BH * Npad * (D / 8);
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  fa_status s;
  if ((s = launch(FA_KERNEL_BWD_PRE, bwd_pre_kernel<D>,
                  dim3((unsigned)std::min<long long>((pre_threads + 255) / 256, (long long)sms() * 8)), dim3(256), 0,
                  st, pp)) != FA_OK)
    return s;
  BwdKVParams kp;
  if ((s = make_tile_map(&kp.q_map, q, bf, 2, hd, N, BH, 64, KV::BM, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&kp.do_map, dO, bf, 2, hd, N, BH, 64, KV::BM, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&kp.k_map, k, bf, 2, hd, N, BH, 64, KV::BN, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&kp.v_map, v, bf, 2, hd, N, BH, 64, KV::BN, sw)) != FA_OK) return s;
  kp.lse2 = lse2;
  kp.dd = dd;
  kp.dqacc = dqacc;
  kp.dk = static_cast<uint16_t*>(dk);
  kp.dv = static_cast<uint16_t*>(dv);
  kp.v = static_cast<const uint16_t*>(v);
  kp.err = err;
  kp.N = N;
  kp.Npad = Npad;
  kp.BH = BH;
  kp.hd = hd;
  kp.scale_log2 = scale * kLog2e;
  kp.scale = scale;
  kp.causal = causal;
  kp.group = causal ? l2_head_group(12.0 * N * D, BH, ((N + KV::BN - 1) / KV::BN) * KV::DSPLIT)
                    : head_group(((N + KV::BN - 1) / KV::BN) * KV::DSPLIT, BH);
  kp.sched = sched;
  kp.qsplit = 1;  // no query-range split: its partial sums would need more scratch
  kp.dkpart = nullptr;
  kp.dvpart = nullptr;
  const long long kv_items = (long long)((N + KV::BN - 1) / KV::BN) * BH * KV::DSPLIT;
  if (kv_items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  kp.items = (int)kv_items;
  const long long kv_grid = std::min<long long>(kv_items, sm_count_cached());
  if ((s = launch(KV::DQ ? FA_KERNEL_BWD_KV5 : FA_KERNEL_BWD_KV7, bwd_kv_kernel<KV, false>, dim3((unsigned)kv_grid),
                  dim3(KV::THREADS), KV::SMEM_BYTES, st, kp)) != FA_OK)
    return s;

  if (five) {
    ConvParams cp{dqacc, static_cast<uint16_t*>(dq), N, Npad, BH, hd, scale};
    const long long groups = (long long)BH * N * hd / 8;  // 8 columns per thread
    return launch(FA_KERNEL_BWD_CONV, bwd_conv_kernel<D>,
                  dim3((unsigned)std::min<long long>((groups + 255) / 256, (long long)sms() * 8)), dim3(256), 0, st,
                  cp);
  }
  BwdQParams qp;
  if ((s = make_tile_map(&qp.q_map, q, bf, 2, hd, N, BH, 64, 128, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&qp.do_map, dO, bf, 2, hd, N, BH, 64, 128, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&qp.k_map, k, bf, 2, hd, N, BH, 64, Q7::BN, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&qp.v_map, v, bf, 2, hd, N, BH, 64, Q7::BN, sw)) != FA_OK) return s;
  qp.lse2 = lse2;
  qp.dd = dd;
  qp.dq = static_cast<uint16_t*>(dq);
  qp.dO = static_cast<const uint16_t*>(dO);
  qp.err = err;
  qp.N = N;
  qp.Npad = Npad;
  qp.BH = BH;
  qp.hd = hd;
  qp.scale_log2 = scale * kLog2e;
  qp.scale = scale;
  qp.causal = causal;
  const int q_tiles = ((N + 127) / 128) * Q7::DQS;
  qp.group = causal ? l2_head_group(12.0 * N * D, BH, q_tiles) : head_group(q_tiles, BH);
  qp.sched = sched;
  qp.ksplit = 1;  // no key-range split: its partial sums would need more scratch
  qp.dqpart = nullptr;
  const long long q_items = (long long)q_tiles * BH;
  if (q_items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  qp.items = (int)q_items;
  const long long q_grid = std::min<long long>(q_items, sm_count_cached());
  return launch(FA_KERNEL_BWD_Q7, bwd_q_kernel<Q7, false>, dim3((unsigned)q_grid), dim3(Q7::THREADS), Q7::SMEM_BYTES,
                st, qp);
}

// Same tile configurations as the workspace-taking backward.
using NKV5_64 = BwdKVCfg<64, 128, true, 1, 2, false>;
using NKV5_128 = BwdKVCfg<128, 64, true, 1, 3, true>;
using NKV7_64 = BwdKVCfg<64, 128, false, 1, 3, false>;
using NKV7_128 = BwdKVCfg<128, 64, false, 1, 4, true>;
using NKV7_192 = BwdKVCfg<192, 64, false, 1, 2, false>;
using NKV7_256 = BwdKVCfg<256, 64, false, 2, 2, false, true, true>;
using NQ7_64 = BwdQCfg<64, 128, 6>;
using NQ7_128 = BwdQCfg<128, 128, 4>;
using NQ7_192 = BwdQCfg<192, 64, 7, true>;
using NQ7_256 = BwdQCfg<256, 64, 5, true>;
using NKV7_384 = BwdKVCfg<384, 32, false, 3, 2, false, true, false>;
using NQ7_384 = BwdQCfg<384, 32, 4, true, 2>;

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                    float scale, int causal, int variant, void* stream) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f) || (causal != 0 && causal != 1)) return FA_ERR_INVALID_ARG;
  if (variant != FA_BWD_AUTO && variant != FA_BWD_5GEMM && variant != FA_BWD_7GEMM) return FA_ERR_INVALID_ARG;
  const int D = padded_head_dim(d);  // 96 runs on zero-padded 128 tiles; 192 on its own (see below)
  if (D == 0) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H > 0x7fffffffLL || (long long)N > 0x7fffffffLL / 2) return FA_ERR_INVALID_ARG;
  if ((long long)B * H * N == 0) return FA_OK;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv};
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) & 15u) return FA_ERR_MISALIGNED;
  const int BH = B * H;
  const int Npad = (N + 127) / 128 * 128;
  // The variant fa_bwd would run; with AUTO, fall back to the 7-GEMM form when
  // only its smaller scratch fits.  Anything beyond the static array is refused.
  bool five = (variant == FA_BWD_AUTO ? fa_bwd_choose(B, H, N, d, causal) : variant) == FA_BWD_5GEMM;
  if (five && D >= 256) return FA_ERR_UNSUPPORTED;
  if (five && scratch_need(BH, Npad, D, true) > kScratchBytes && variant == FA_BWD_AUTO) five = false;
  if (scratch_need(BH, Npad, D, five) > kScratchBytes) return FA_ERR_WORKSPACE;
  unsigned char* base = scratch_address();
  if (!base) return FA_ERR_LAUNCH;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (D) {
    case 64:
      return five ? run<NKV5_64, NQ7_64, 64>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal, true, base, st)
                  : run<NKV7_64, NQ7_64, 64>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal, false, base, st);
    case 128:
      return five ? run<NKV5_128, NQ7_128, 128>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal, true, base,
                                                st)
                  : run<NKV7_128, NQ7_128, 128>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal, false, base,
                                                st);
    case 384:
      return run<NKV7_384, NQ7_384, 384>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal, false, base, st);
    default:
      if (d == 192)
        return run<NKV7_192, NQ7_192, 256>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal, false, base, st);
      return run<NKV7_256, NQ7_256, 256>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal, false, base, st);
  }
}

// The error word of the static array: read (and cleared) without allocating.
extern "C" fa_status fa_bwd_noalloc_device_error(void* stream, int* site) {
  if (site) *site = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda_error(e);
  unsigned char* base = scratch_address();
  if (!base) return FA_ERR_LAUNCH;
  int h[2] = {0, 0};
  e = cudaMemcpy(h, base, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return record_cuda_error(e);
  if (h[0] == 0) return FA_OK;
  if (site) *site = h[1];
  e = cudaMemset(base, 0, sizeof(h));
  if (e != cudaSuccess) return record_cuda_error(e);
  return FA_ERR_DEVICE_TIMEOUT;
}

extern "C" fa_status fa_bwd_noalloc_watchdog_selftest(void* stream) {
  unsigned char* base = scratch_address();
  if (!base) return FA_ERR_LAUNCH;
  return launch_watchdog_selftest(reinterpret_cast<int*>(base), static_cast<cudaStream_t>(stream));
}
