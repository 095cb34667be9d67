// Backward launchers: workspace carving, tile configurations and TMA descriptors.
#include "bwd.cuh"
#include <algorithm>
#include <type_traits>

#include "host.h"

namespace fa {
namespace {

// dK/dV kernel configurations <d, query rows per step, with dQ, d split, query stages, separate P/dS>.
// d = 128 5-GEMM: bulk dQ reductions from a shared-memory tile measured faster than per-element
// or 16-byte reductions straight from registers, worth giving up one query stage.
// d = 64 5-GEMM: 128 query columns per step over two compute warpgroups, each packing its P^T / dS^T
// into its own S^T / dP^T columns.
using KV5_64 = BwdKVCfg<64, 128, true, 1, 2, false>;
using KV5_128 = BwdKVCfg<128, 64, true, 1, 3, true>;
using KV7_64 = BwdKVCfg<64, 128, false, 1, 3, false>;
using KV7_128 = BwdKVCfg<128, 64, false, 1, 4, true>;
// d = 192: dV and dK for all 192 columns fit TMEM next to S and dP, so no d split.
using KV7_192 = BwdKVCfg<192, 64, false, 1, 2, false>;
// d = 256: V in TMEM, and the outputs split (a dV item and a dK item per key tile, each with one
// 256-column accumulator).
using KV7_256 = BwdKVCfg<256, 64, false, 2, 2, false, true, true>;
// dQ kernel configurations <d, keys per tile, K/V ring slots>.
using Q7_64 = BwdQCfg<64, 128, 6>;
using Q7_128 = BwdQCfg<128, 128, 4>;
using Q7_192 = BwdQCfg<192, 64, 7, true>;
using Q7_256 = BwdQCfg<256, 64, 5, true>;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct Workspace {
  float* lse2;
  float* dd;
  float* dqacc;
  int* sched;  // work-item counters, in the workspace's last 256 bytes
};

Workspace carve(void* ws, int BH, int Npad, int d, bool with_dq) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  const size_t rows = (size_t)BH * Npad;
  Workspace w;
  w.lse2 = reinterpret_cast<float*>(b);
  w.dd = reinterpret_cast<float*>(b + align256(4 * rows));
  w.dqacc = with_dq ? reinterpret_cast<float*>(b + 2 * align256(4 * rows)) : nullptr;
  w.sched = reinterpret_cast<int*>(b + 2 * align256(4 * rows) + (with_dq ? 4 * rows * (size_t)d : 0));
  return w;
}

int sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

template <int D>
fa_status run_pre(const void* o, const void* dO, const float* lse, const Workspace& w, int BH, int N, int Npad,
                  int hd, cudaStream_t st) {
  PreParams p{static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dO), lse, w.lse2, w.dd, w.dqacc,
              N, Npad, BH, hd, w.sched};
  const long long threads = (long long)BH * Npad * (D / 8);
  const long long blocks = std::min<long long>((threads + 255) / 256, (long long)sm_count() * 8);
  return launch(FA_KERNEL_BWD_PRE, bwd_pre_kernel<D>, dim3((unsigned)blocks), dim3(256), 0, st, p);
}

template <int D>
fa_status run_conv(const Workspace& w, void* dq, int BH, int N, int Npad, int hd, float scale, cudaStream_t st) {
  ConvParams p{w.dqacc, static_cast<uint16_t*>(dq), N, Npad, BH, hd, scale};
  const long long groups = (long long)BH * N * hd / 8;  // 8 columns per thread
  const long long blocks = std::min<long long>((groups + 255) / 256, (long long)sm_count() * 8);
  return launch(FA_KERNEL_BWD_CONV, bwd_conv_kernel<D>, dim3((unsigned)blocks), dim3(256), 0, st, p);
}

template <class C>
fa_status run_kv(const void* q, const void* k, const void* v, const void* dO, const Workspace& w, void* dk,
                 void* dv, int BH, int N, int Npad, int hd, float scale, int causal, cudaStream_t st) {
  BwdKVParams p;
  fa_status s;
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if ((s = make_tile_map(&p.q_map, q, bf, 2, hd, N, BH, 64, C::BM, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&p.do_map, dO, bf, 2, hd, N, BH, 64, C::BM, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&p.k_map, k, bf, 2, hd, N, BH, 64, C::BN, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&p.v_map, v, bf, 2, hd, N, BH, 64, C::BN, sw)) != FA_OK) return s;
  p.lse2 = w.lse2;
  p.dd = w.dd;
  p.dqacc = w.dqacc;
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  p.v = static_cast<const uint16_t*>(v);
  p.err = device_error_word();
  if (!p.err) return record_cuda_error(cudaErrorMemoryAllocation);
  p.N = N;
  p.Npad = Npad;
  p.BH = BH;
  p.hd = hd;
  p.scale_log2 = scale * kLog2e;
  p.scale = scale;
  p.causal = causal;
  p.group = causal ? l2_head_group(12.0 * N * C::D, BH, ((N + C::BN - 1) / C::BN) * C::DSPLIT)
                   : head_group(((N + C::BN - 1) / C::BN) * C::DSPLIT, BH);
  p.sched = w.sched;
  const long long items = (long long)((N + C::BN - 1) / C::BN) * BH * C::DSPLIT;
  if (items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.items = (int)items;
  // Persistent grid: one CTA per SM (one fits per SM), each walking its items.
  const long long grid = std::min<long long>(items, sm_count_cached());
  return launch(C::DQ ? FA_KERNEL_BWD_KV5 : FA_KERNEL_BWD_KV7, bwd_kv_kernel<C>, dim3((unsigned)grid),
                dim3(C::THREADS), C::SMEM_BYTES, st, p);
}

template <class C>
fa_status run_q(const void* q, const void* k, const void* v, const void* dO, const Workspace& w, void* dq, int BH,
                int N, int Npad, int hd, float scale, int causal, cudaStream_t st) {
  BwdQParams p;
  fa_status s;
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if ((s = make_tile_map(&p.q_map, q, bf, 2, hd, N, BH, 64, 128, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&p.do_map, dO, bf, 2, hd, N, BH, 64, 128, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&p.k_map, k, bf, 2, hd, N, BH, 64, C::BN, sw)) != FA_OK) return s;
  if ((s = make_tile_map(&p.v_map, v, bf, 2, hd, N, BH, 64, C::BN, sw)) != FA_OK) return s;
  p.lse2 = w.lse2;
  p.dd = w.dd;
  p.dq = static_cast<uint16_t*>(dq);
  p.dO = static_cast<const uint16_t*>(dO);
  p.err = device_error_word();
  if (!p.err) return record_cuda_error(cudaErrorMemoryAllocation);
  p.N = N;
  p.Npad = Npad;
  p.BH = BH;
  p.hd = hd;
  p.scale_log2 = scale * kLog2e;
  p.scale = scale;
  p.causal = causal;
  p.group = causal ? l2_head_group(12.0 * N * C::D, BH, (N + 127) / 128) : head_group((N + 127) / 128, BH);
  p.sched = w.sched;
  const long long items = (long long)((N + 127) / 128) * BH;
  if (items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.items = (int)items;
  // Persistent grid: one CTA per SM, each claiming work items.
  const long long grid = std::min<long long>(items, sm_count_cached());
  return launch(FA_KERNEL_BWD_Q7, bwd_q_kernel<C>, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, st, p);
}

template <int D, class KV5, class KV7, class Q7>
fa_status run_d(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                void* dq, void* dk, void* dv, int BH, int N, int hd, float scale, int causal, int variant, void* ws,
                cudaStream_t st) {
  const int Npad = (N + 127) / 128 * 128;
  const bool five = variant == FA_BWD_5GEMM;
  const Workspace w = carve(ws, BH, Npad, D, five);
  fa_status s = run_pre<D>(o, dO, lse, w, BH, N, Npad, hd, st);
  if (s != FA_OK) return s;
  if (five) {
    if constexpr (!std::is_same<KV5, void>::value) {
      if ((s = run_kv<KV5>(q, k, v, dO, w, dk, dv, BH, N, Npad, hd, scale, causal, st)) != FA_OK) return s;
      return run_conv<D>(w, dq, BH, N, Npad, hd, scale, st);
    }
    return FA_ERR_UNSUPPORTED;
  }
  if ((s = run_kv<KV7>(q, k, v, dO, w, dk, dv, BH, N, Npad, hd, scale, causal, st)) != FA_OK) return s;
  return run_q<Q7>(q, k, v, dO, w, dq, BH, N, Npad, hd, scale, causal, st);
}

}  // namespace

// d = 96 runs the d = 128 kernels on zero-padded tiles (TMA reads the columns
// past d as zeros; nothing past d is stored).  d = 192 has its own dK/dV and dQ
// kernels; its preprocess is the d = 256 one (which reads only d columns).
fa_status run_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                  void* dq, void* dk, void* dv, int BH, int N, int d, float scale, int causal, int variant,
                  void* workspace, cudaStream_t st) {
  if (d == 192)
    return run_d<256, void, KV7_192, Q7_192>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal, variant,
                                             workspace, st);
  switch (padded_head_dim(d)) {
    case 64:
      return run_d<64, KV5_64, KV7_64, Q7_64>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal, variant,
                                              workspace, st);
    case 128:
      return run_d<128, KV5_128, KV7_128, Q7_128>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal,
                                                  variant, workspace, st);
    case 256:
      return run_d<256, void, KV7_256, Q7_256>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal, variant,
                                               workspace, st);
  }
  return FA_ERR_UNSUPPORTED;
}

bool bwd_supported(int d, int variant) {
  const int D = padded_head_dim(d);
  if (variant == FA_BWD_7GEMM) return D != 0;
  if (variant == FA_BWD_5GEMM) return D == 64 || D == 128;
  return false;
}

int bwd_launch_count(int, int) { return 3; }

}  // namespace fa
