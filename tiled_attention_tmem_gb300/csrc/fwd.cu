// Forward launcher: tile configuration per head dimension and TMA descriptors.
#include "fwd.cuh"
#include <algorithm>

#include "host.h"

namespace fa {
namespace {

// Per head dimension: query tiles per CTA, keys per tile, K/V ring depth.
//  d = 64 : 2 x 128 query rows, 128 keys, 6 stages (Q 32 KiB + ring 96 KiB)
//  d = 128: 2 x 128 query rows, 128 keys, 4 stages (Q 64 KiB + ring 128 KiB)
//  d = 192: 1 x 128 query rows, 64 keys, 8 stages, Q in TMEM (ring 192 KiB)
//  d = 256: 1 x 128 query rows, 64 keys, 6 stages, Q in TMEM (ring 192 KiB)
//  d = 384: 1 x 128 query rows, 64 keys, 2 stages, Q in shared memory
// d = 96 runs the d = 128 kernel: the TMA boxes read columns past d as zeros,
// which leave S = QK^T unchanged and give zero output columns that are not
// stored.
using Fwd64 = FwdCfg<64, 2, 128, 6>;
using Fwd128 = FwdCfg<128, 2, 128, 4>;
using Fwd192 = FwdCfg<192, 1, 64, 8, true>;
using Fwd256 = FwdCfg<256, 1, 64, 6, true>;
// d = 384: 1 x 128 query rows, 64 keys, Q in shared memory (96 KiB) with S
// double-buffered in TMEM next to the 384-column O (512 columns), two K/V slots
// of 48 KiB.
using Fwd384 = FwdCfg<384, 1, 64, 2, false, true>;

template <class C>
fa_status run(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int N, int d,
              float scale, int causal, int splits, void* workspace, cudaStream_t st) {
  FwdParams p;
  fa_status s;
  if ((s = make_tile_map(&p.q_map, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B)) != FA_OK)
    return s;
  if ((s = make_tile_map(&p.k_map, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64, C::BN,
                         CU_TENSOR_MAP_SWIZZLE_128B)) != FA_OK)
    return s;
  if ((s = make_tile_map(&p.v_map, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64, C::BN,
                         CU_TENSOR_MAP_SWIZZLE_128B)) != FA_OK)
    return s;
  p.q = static_cast<const uint16_t*>(q);
  p.o = static_cast<uint16_t*>(o);
  p.dv = d;
  p.lse = lse;
  p.err = device_error_word();
  if (!p.err) return record_cuda_error(cudaErrorMemoryAllocation);
  p.N = N;
  p.BH = BH;
  p.scale_log2 = scale * kLog2e;
  p.causal = causal;
  const int n_qblk = (N + 128 * C::NQ - 1) / (128 * C::NQ);
  // Causal: heaviest query blocks first inside groups of heads whose K and V
  // (4 N d bytes each) stay in L2.
  p.group = causal ? l2_head_group(4.0 * N * d, BH, n_qblk) : head_group(n_qblk, BH);
  const long long items = (long long)n_qblk * BH * splits;
  if (items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.items = (int)items;
  p.splits = splits;
  p.opart = nullptr;
  p.lpart = nullptr;
  const long long rows = (long long)BH * N;
  if (splits > 1) {
    p.opart = static_cast<float*>(workspace);
    p.lpart = reinterpret_cast<float*>(static_cast<char*>(workspace) + splitkv_lse_offset(BH, N, d, splits));
  }
  // Persistent grid: one CTA per SM (shared memory allows no more), each walking
  // its share of the work items.
  const long long grid = std::min<long long>(items, sm_count_cached());
  if (splits == 1)
    return launch(FA_KERNEL_FWD, fwd_kernel<C, false>, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES,
                  st, p);
  fa_status s2 =
      launch(FA_KERNEL_FWD, fwd_kernel<C, true>, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, st, p);
  if (s2 != FA_OK) return s2;
  FwdMergeParams mp;
  mp.opart = p.opart;
  mp.lpart = p.lpart;
  mp.o = p.o;
  mp.lse = lse;
  mp.err = p.err;
  mp.rows = rows;
  mp.dv = d;
  mp.splits = splits;
  const long long threads = rows * (d / 8);
  const long long blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  return launch(FA_KERNEL_FWD_MERGE, fwd_merge_kernel, dim3((unsigned)blocks), dim3(256), 0, st, mp);
}

}  // namespace

fa_status run_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int N,
                  int d, float scale, int causal, int splits, void* workspace, cudaStream_t st) {
  switch (d) {
    case 64: return run<Fwd64>(q, k, v, o, lse, BH, N, d, scale, causal, splits, workspace, st);
    case 96:
    case 128: return run<Fwd128>(q, k, v, o, lse, BH, N, d, scale, causal, splits, workspace, st);
    case 192: return run<Fwd192>(q, k, v, o, lse, BH, N, d, scale, causal, splits, workspace, st);
    case 256: return run<Fwd256>(q, k, v, o, lse, BH, N, d, scale, causal, splits, workspace, st);
    case 384: return run<Fwd384>(q, k, v, o, lse, BH, N, d, scale, causal, splits, workspace, st);
  }
  return FA_ERR_UNSUPPORTED;
}

size_t splitkv_lse_offset(int BH, int N, int d, int splits) {
  const size_t o_bytes = (size_t)splits * BH * N * d * sizeof(float);
  return (o_bytes + 255) / 256 * 256;
}

size_t splitkv_workspace_bytes(int BH, int N, int d, int splits) {
  if (splits <= 1) return 0;
  const size_t l_bytes = (size_t)splits * BH * N * sizeof(float);
  return splitkv_lse_offset(BH, N, d, splits) + (l_bytes + 255) / 256 * 256;
}

int choose_splits(int BH, int N, int d, int causal) {
  // Cost model in microseconds, fitted to a GB300 sweep of the split count over
  // one to four long heads at d = 64, 128, 192 and 256.  The persistent grid runs
  // the parts in ceil(parts / SMs) rounds, and cannot finish before the heaviest
  // part (under the causal mask the last query block sees every key tile); a part
  // costs its key steps plus about two steps of setup and epilogue; a key step
  // takes the larger of 1.2x its MMA cycles and 1.3k cycles (the softmax
  // latency) at about 1.9 GHz.  Splitting adds the merge kernel: about 6 us plus
  // its fp32 reads and bf16 writes at about 6 TB/s.
  const int rows_item = d <= 128 ? 256 : 128;
  const int bn = d <= 128 ? 128 : 64;
  const int dk = d <= 64 ? 64 : d <= 128 ? 128 : d;
  const long long items = (long long)BH * ((N + rows_item - 1) / rows_item);
  const int tiles = (N + bn - 1) / bn;
  const double sms = sm_count_cached();
  const double step_us = std::max(1.2 * 4.0 * rows_item * bn * dk / 8192.0, 1300.0) / 1.9e3;
  const double mean = causal ? (tiles + 1) / 2.0 : tiles;  // key tiles of the mean item
  auto cost = [&](int s) {
    const double rounds = std::ceil(items * (double)s / sms);
    double us = std::max(rounds * (mean / s + 2.0), (double)tiles / s + 2.0) * step_us;
    if (s > 1) us += 6.0 + (double)BH * N * (4.0 * s * (d + 1) + 2.0 * d + 4.0) / 6.0e6;
    return us;
  };
  int best = 1;
  double best_us = cost(1);
  for (int s = 2; s <= kMaxSplits && tiles / s >= 2; ++s) {
    const double us = cost(s);
    if (us < 0.97 * best_us) {
      best = s;
      best_us = us;
    }
  }
  return best;
}

int fwd_launch_count(int) { return 1; }

}  // namespace fa
