// Backward launchers: workspace carving, tile configurations and TMA descriptors.
#include "bwd.cuh"
#include <algorithm>
#include <atomic>
#include <cmath>
#include <map>
#include <mutex>
#include <tuple>
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
// d = 384: dV and dK cut into three column parts of 128, one work item each (every item
// recomputes S^T and dP^T), 32 queries per step, V in TMEM: 32 + 32 + 128 + 128 + 192 = 512
// TMEM columns next to a 96 KiB K tile and two 48 KiB query stages.
using KV7_384 = BwdKVCfg<384, 32, false, 3, 2, false, true, false>;
// dQ kernel configurations <d, keys per tile, K/V ring slots>.
using Q7_64 = BwdQCfg<64, 128, 6>;
using Q7_128 = BwdQCfg<128, 128, 4>;
using Q7_192 = BwdQCfg<192, 64, 7, true>;
using Q7_256 = BwdQCfg<256, 64, 5, true>;
// d = 384: two dQ column parts of 192 per query tile (one work item each), dO in TMEM,
// 32-key tiles, four K/V slots of 24 KiB next to the 96 KiB Q tile.
using Q7_384 = BwdQCfg<384, 32, 4, true, 2>;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct Workspace {
  float* lse2;
  float* dd;
  float* dqacc;
  float* dkpart;  // query-range split: fp32 partial dK, dV [qsplit][BH][Npad][d]
  float* dvpart;
  float* dqpart;  // key-range split of the dQ kernel: fp32 partial dQ [ksplit][BH][Npad][d]
  int* sched;  // work-item counters, in the workspace's last 256 bytes
};

Workspace carve(void* ws, int BH, int Npad, int d, bool with_dq, int qsplit, int ksplit) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  const size_t rows = (size_t)BH * Npad;
  Workspace w;
  w.lse2 = reinterpret_cast<float*>(b);
  w.dd = reinterpret_cast<float*>(b + align256(4 * rows));
  size_t off = 2 * align256(4 * rows);
  w.dqacc = with_dq ? reinterpret_cast<float*>(b + off) : nullptr;
  off += with_dq ? 4 * rows * (size_t)d : 0;
  w.dkpart = w.dvpart = nullptr;
  if (qsplit > 1) {
    const size_t part_bytes = 4 * (size_t)qsplit * rows * d;
    w.dkpart = reinterpret_cast<float*>(b + off);
    w.dvpart = reinterpret_cast<float*>(b + off + part_bytes);
    off += 2 * part_bytes;
  }
  w.dqpart = nullptr;
  if (ksplit > 1) {
    w.dqpart = reinterpret_cast<float*>(b + off);
    off += 4 * (size_t)ksplit * rows * d;
  }
  w.sched = reinterpret_cast<int*>(b + off);
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
                 void* dv, int BH, int N, int Npad, int hd, float scale, int causal, int qsplit, cudaStream_t st) {
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
  const int tiles = ((N + C::BN - 1) / C::BN) * C::DSPLIT * qsplit;
  p.group = causal ? l2_head_group(12.0 * N * C::D, BH, tiles) : head_group(tiles, BH);
  p.sched = w.sched;
  p.qsplit = qsplit;
  p.dkpart = w.dkpart;
  p.dvpart = w.dvpart;
  const long long items = (long long)tiles * BH;
  if (items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.items = (int)items;
  // Persistent grid: one CTA per SM (one fits per SM), each walking its items.
  const long long grid = std::min<long long>(items, sm_count_cached());
  const int kind = C::DQ ? FA_KERNEL_BWD_KV5 : FA_KERNEL_BWD_KV7;
  // Few work items (about four per SM or fewer): the instantiation with the query
  // split and staggered query-tile walks.
  const bool few = qsplit > 1 || (long long)((N + C::BN - 1) / C::BN) * C::DSPLIT * BH < 4LL * sm_count_cached();
  if (!few)
    return launch(kind, bwd_kv_kernel<C, false>, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, st, p);
  fa_status s2 = launch(kind, bwd_kv_kernel<C, true>, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, st, p);
  if (s2 != FA_OK || qsplit <= 1) return s2;
  KVSumParams sp{w.dkpart, w.dvpart, static_cast<uint16_t*>(dk), static_cast<uint16_t*>(dv), p.err,
                 N, Npad, BH, hd, C::D, qsplit, scale};
  const long long threads = (long long)BH * N * (hd / 8);
  return launch(FA_KERNEL_BWD_KVSUM, bwd_kvsum_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, st, sp);
}

template <class C>
fa_status run_q(const void* q, const void* k, const void* v, const void* dO, const Workspace& w, void* dq, int BH,
                int N, int Npad, int hd, float scale, int causal, int ksplit, cudaStream_t st) {
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
  const int tiles = ((N + 127) / 128) * C::DQS * ksplit;
  p.group = causal ? l2_head_group(12.0 * N * C::D, BH, tiles) : head_group(tiles, BH);
  p.sched = w.sched;
  p.ksplit = ksplit;
  p.dqpart = w.dqpart;
  const long long items = (long long)tiles * BH;
  if (items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.items = (int)items;
  // Persistent grid: one CTA per SM, each claiming work items.
  const long long grid = std::min<long long>(items, sm_count_cached());
  if (ksplit <= 1)
    return launch(FA_KERNEL_BWD_Q7, bwd_q_kernel<C, false>, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES,
                  st, p);
  fa_status s2 =
      launch(FA_KERNEL_BWD_Q7, bwd_q_kernel<C, true>, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, st, p);
  if (s2 != FA_OK) return s2;
  QSumParams sp{w.dqpart, static_cast<uint16_t*>(dq), p.err, N, Npad, BH, hd, C::D, ksplit, scale};
  const long long threads = (long long)BH * N * (hd / 8);
  return launch(FA_KERNEL_BWD_QSUM, bwd_qsum_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, st, sp);
}

template <int D, class KV5, class KV7, class Q7>
fa_status run_d(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                void* dq, void* dk, void* dv, int BH, int N, int hd, float scale, int causal, int variant, void* ws,
                cudaStream_t st) {
  const int Npad = (N + 127) / 128 * 128;
  const bool five = variant == FA_BWD_5GEMM;
  const int qsplit = choose_qsplit(BH, N, hd, causal, variant);
  const int ksplit = five ? 1 : choose_ksplit(BH, N, hd, causal, variant);
  const Workspace w = carve(ws, BH, Npad, D, five, qsplit, ksplit);
  fa_status s = run_pre<D>(o, dO, lse, w, BH, N, Npad, hd, st);
  if (s != FA_OK) return s;
  if (five) {
    if constexpr (!std::is_same<KV5, void>::value) {
      if ((s = run_kv<KV5>(q, k, v, dO, w, dk, dv, BH, N, Npad, hd, scale, causal, qsplit, st)) != FA_OK) return s;
      return run_conv<D>(w, dq, BH, N, Npad, hd, scale, st);
    }
    return FA_ERR_UNSUPPORTED;
  }
  if ((s = run_kv<KV7>(q, k, v, dO, w, dk, dv, BH, N, Npad, hd, scale, causal, qsplit, st)) != FA_OK) return s;
  return run_q<Q7>(q, k, v, dO, w, dq, BH, N, Npad, hd, scale, causal, ksplit, st);
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
  if (d == 384)
    return run_d<384, void, KV7_384, Q7_384>(q, k, v, o, dO, lse, dq, dk, dv, BH, N, d, scale, causal, variant,
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

int bwd_launch_count(int BH, int N, int d, int causal, int variant) {
  return 3 + (choose_qsplit(BH, N, d, causal, variant) > 1 ? 1 : 0) +
         (choose_ksplit(BH, N, d, causal, variant) > 1 ? 1 : 0);
}

size_t bwd_split_bytes(int BH, int N, int d, int causal, int variant) {
  const int qsplit = choose_qsplit(BH, N, d, causal, variant);
  const int ksplit = choose_ksplit(BH, N, d, causal, variant);
  const size_t slab = 4 * (size_t)BH * ((size_t)(N + 127) / 128 * 128) * (size_t)padded_head_dim(d);
  return (qsplit > 1 ? 2 * (size_t)qsplit * slab : 0) + (ksplit > 1 ? (size_t)ksplit * slab : 0);
}

namespace {
int choose_qsplit_uncached(int BH, int N, int d, int causal, int variant) {
  const int D = padded_head_dim(d);
  if (D == 0 || BH <= 0 || N <= 0) return 1;
  // d = 256 (7-GEMM): a dV item and a dK item per key tile; d = 384: three column parts.
  const int dsplit = (variant != FA_BWD_5GEMM && D == 256) ? 2 : D == 384 ? 3 : 1;
  const double items = (double)((N + 127) / 128) * dsplit * BH;
  const double sms = sm_count_cached();
  if (items >= 2.0 * sms) return 1;
  const int cap = std::max(1, std::min(8, N / 512));
  long parts;
  if (causal)
    parts = std::lround(3.0 * sms / items);
  else if (items <= 0.85 * sms)
    parts = std::max(2L, std::lround(0.85 * sms / items));
  else
    parts = 1;
  return (int)std::max(1L, std::min((long)cap, parts));
}
std::mutex g_qsplit_mutex;
std::map<std::tuple<int, int, int, int, int, int>, int> g_qsplit_cache;
std::atomic<int> g_qsplit_forced{0};
std::atomic<int> g_ksplit_forced{0};

// The dQ kernel's key split takes the query split's rule (below) over its own
// work items: query tiles x dQ column parts x heads.
int choose_ksplit_uncached(int BH, int N, int d, int causal) {
  const int D = padded_head_dim(d);
  if (D == 0 || BH <= 0 || N <= 0) return 1;
  const double items = (double)((N + 127) / 128) * (D == 384 ? 2 : 1) * BH;
  const double sms = sm_count_cached();
  if (items >= 2.0 * sms) return 1;
  const int cap = std::max(1, std::min(8, N / 512));
  long parts;
  if (causal)
    parts = std::lround(3.0 * sms / items);
  else if (items <= 0.85 * sms)
    parts = std::max(2L, std::lround(0.85 * sms / items));
  else
    parts = 1;
  return (int)std::max(1L, std::min((long)cap, parts));
}
}  // namespace

void force_qsplit(int parts) { g_qsplit_forced.store(parts); }
void force_ksplit(int parts) { g_ksplit_forced.store(parts); }

// Key parts per query tile of the 7-GEMM dQ kernel (1 for the 5-GEMM form, which
// has no dQ kernel).  Cheap enough to compute per call.
int choose_ksplit(int BH, int N, int d, int causal, int variant) {
  if (variant == FA_BWD_5GEMM) return 1;
  if (const int forced = g_ksplit_forced.load()) return forced;
  return choose_ksplit_uncached(BH, N, d, causal);
}

// Query parts per key tile for the dK/dV kernel.  A persistent grid finishes no
// earlier than its longest work item; with few heads there are fewer key tiles
// than SMs, and under the causal mask the first key tile of a head sees every
// query tile, so splitting the query range shortens the critical path at the
// price of more item changes and a summing kernel.  (Without the mask, one long
// item per SM of a single head also ran up to twice slower per step than the
// same work cut in two parts, in some runs and not in others.)  The rule is
// fitted to two GB300 sweeps of the part count (1, 2, 3, 4, 6, 8) over one to
// sixteen heads, N = 2048 to 16384, head dims 64 to 384 and both masks, 128
// measurements (geometric-mean time 1.07x the best measured part count,
// against 1.37x without splitting):
//   - no split once the items fill two waves of SMs;
//   - causal: about three items per SM;
//   - no mask: up to 0.85 items per SM, about one item per SM and at least two
//     parts; none above;
//   - at least 512 query rows per part, at most 8 parts.
int choose_qsplit(int BH, int N, int d, int causal, int variant) {
  if (const int forced = g_qsplit_forced.load()) return forced;
  const auto key = std::make_tuple(BH, N, d, causal, variant, sm_count_cached());
  {
    std::lock_guard<std::mutex> lock(g_qsplit_mutex);
    auto it = g_qsplit_cache.find(key);
    if (it != g_qsplit_cache.end()) return it->second;
  }
  const int q = choose_qsplit_uncached(BH, N, d, causal, variant);
  std::lock_guard<std::mutex> lock(g_qsplit_mutex);
  if (g_qsplit_cache.size() > 4096) g_qsplit_cache.clear();
  g_qsplit_cache[key] = q;
  return q;
}

}  // namespace fa
