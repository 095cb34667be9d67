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
// d = 96 runs the d = 128 kernel: the TMA boxes read columns past d as zeros,
// which leave S = QK^T unchanged and give zero output columns that are not
// stored.
using Fwd64 = FwdCfg<64, 2, 128, 6>;
using Fwd128 = FwdCfg<128, 2, 128, 4>;
using Fwd192 = FwdCfg<192, 1, 64, 8, true>;
using Fwd256 = FwdCfg<256, 1, 64, 6, true>;

template <class C>
fa_status run(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int N, int d,
              float scale, int causal, cudaStream_t st) {
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
  const long long items = (long long)n_qblk * BH;
  if (items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.items = (int)items;
  // Persistent grid: one CTA per SM (shared memory allows no more), each walking
  // its share of the work items.
  const long long grid = std::min<long long>(items, sm_count_cached());
  return launch(FA_KERNEL_FWD, fwd_kernel<C>, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, st, p);
}

}  // namespace

fa_status run_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int N,
                  int d, float scale, int causal, cudaStream_t st) {
  switch (d) {
    case 64: return run<Fwd64>(q, k, v, o, lse, BH, N, d, scale, causal, st);
    case 96:
    case 128: return run<Fwd128>(q, k, v, o, lse, BH, N, d, scale, causal, st);
    case 192: return run<Fwd192>(q, k, v, o, lse, BH, N, d, scale, causal, st);
    case 256: return run<Fwd256>(q, k, v, o, lse, BH, N, d, scale, causal, st);
  }
  return FA_ERR_UNSUPPORTED;
}

int fwd_launch_count(int) { return 1; }

}  // namespace fa
