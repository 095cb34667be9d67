// Fused attention backward.
//
// Method: the backward recomputes P from the per-row log-sum-exp kept by the
// forward instead of storing it ("ELI5: FlashAttention", recomputation), forms
// D_i = dO_i . O_i, and then
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  dK = scale dS^T Q,  dQ = scale dS K.
// Two variants, as debated in "Potential algorithmic improvements for backward
// pass" (FlashAttention issue 1172):
//   5-GEMM: one kernel per K/V tile runs S, dP, dV, dK and dQ; each K/V tile's
//           dQ contribution is added into an fp32 accumulator in global memory
//           (bulk asynchronous reductions), then converted to bf16.
//   7-GEMM: the dK/dV kernel runs S, dP, dV, dK; a second kernel walks each
//           query tile over the K/V tiles like the forward and runs S, dP, dQ.
//           No atomics, so the result is bitwise reproducible.
//
// Workspace (fp32, rows padded to Npad = 128 * ceil(N / 128) per head):
//   lse2[bh][Npad]  -LSE * log2(e) for valid rows, -inf for padding rows
//   dd[bh][Npad]    -D for valid rows, 0 for padding rows
//   (stored negated so P = exp2(S c + lse2) and dS = P (dP + dd) are single
//   packed FMA / add instructions)
//   dqacc[bh][Npad][d] (5-GEMM) with the 16-byte chunks of row i permuted by
//                   chunk ^ (i % 8), which makes the staging writes of both
//                   dQ orientations free of shared-memory bank conflicts.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"

namespace fa {

__device__ __forceinline__ int dq_swz(int i, int c) { return ((((c >> 2) ^ (i & 7))) << 2) | (c & 3); }

__device__ __forceinline__ void wait_drain_bwd(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_test(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ----------------------------------------------------------------- preprocess
// One group of G threads per row (G = d/8 up to 32, 16 at d = 384), each
// taking CH chunks of 8 columns: D_i = sum_c dO_ic O_ic (fp32), the
// log2-domain LSE (both stored negated), and (5-GEMM) zeroing of the row's fp32
// dQ accumulator.
struct PreParams {
  const uint16_t* o;
  const uint16_t* dO;
  const float* lse;
  float* lse2;
  float* dd;
  float* dqacc;  // nullptr for the 7-GEMM variant
  int N, Npad, BH, dv;  // dv: head dim of O and dO (<= D; the kernel's D covers padded columns)
  int* sched;    // work-item counters of the following kernels, zeroed here
};

template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const PreParams p) {
  grid_dep_wait();
  constexpr int G = D / 8 <= 32 ? D / 8 : 16;  // threads per row (a power of two)
  constexpr int CH = D / 8 / G;                // 8-column chunks per thread
  static_assert(G * CH * 8 == D && (G & (G - 1)) == 0, "preprocess row split");
  const long long rows = (long long)p.BH * p.Npad;
  const int sub = threadIdx.x % G;
  for (long long row = ((long long)blockIdx.x * 256 + threadIdx.x) / G; row < rows;
       row += (long long)gridDim.x * 256 / G) {
    const int bh = (int)(row / p.Npad);
    const int i = (int)(row % p.Npad);
    float acc = 0.f;
#pragma unroll
    for (int ch = 0; ch < CH; ++ch) {
      const int c = (ch * G + sub) * 8;
      if (i < p.N && c < p.dv) {
        const size_t off = ((size_t)bh * p.N + i) * p.dv + c;
        const uint4 a = *reinterpret_cast<const uint4*>(p.o + off);
        const uint4 b = *reinterpret_cast<const uint4*>(p.dO + off);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc = fmaf(__uint_as_float(av[e] << 16), __uint_as_float(bv[e] << 16), acc);
          acc = fmaf(__uint_as_float(av[e] & 0xffff0000u), __uint_as_float(bv[e] & 0xffff0000u), acc);
        }
      }
    }
#pragma unroll
    for (int w = G / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w, G);
    if (sub == 0) {
      p.dd[row] = -acc;
      p.lse2[row] = i < p.N ? -(p.lse[(size_t)bh * p.N + i] * kLog2e) : -INFINITY;
    }
    if (p.sched && row == 0 && sub < 4) p.sched[sub] = 0;
    if (p.dqacc) {
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) {
        float4* z = reinterpret_cast<float4*>(p.dqacc + (size_t)row * D + (ch * G + sub) * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// --------------------------------------------------------------- dQ convert
struct ConvParams {
  const float* dqacc;  // [bh][Npad][D], D = padded head dim
  uint16_t* dq;        // [bh][N][dv]
  int N, Npad, BH, dv;
  float scale;
};

template <int D>
__global__ void __launch_bounds__(256) bwd_conv_kernel(const ConvParams p) {
  grid_dep_wait();
  // Each thread converts 8 consecutive columns (two 16-byte loads, one 16-byte
  // store); two groups per iteration keep four loads in flight.
  const long long n8 = (long long)p.BH * p.N * p.dv / 8;
  const long long stride = (long long)gridDim.x * 256;
  auto convert = [&](long long g) {
    const long long e = g * 8;
    const int c = (int)(e % p.dv);
    const long long rowg = e / p.dv;  // bh * N + i
    const int bh = (int)(rowg / p.N);
    const int i = (int)(rowg % p.N);
    const float* row = p.dqacc + ((size_t)bh * p.Npad + i) * D;
    const float4 a = *reinterpret_cast<const float4*>(row + dq_swz(i, c));
    const float4 b = *reinterpret_cast<const float4*>(row + dq_swz(i, c + 4));
    uint4 out;
    out.x = pack_bf16(a.x * p.scale, a.y * p.scale);
    out.y = pack_bf16(a.z * p.scale, a.w * p.scale);
    out.z = pack_bf16(b.x * p.scale, b.y * p.scale);
    out.w = pack_bf16(b.z * p.scale, b.w * p.scale);
    *reinterpret_cast<uint4*>(p.dq + e) = out;
  };
  long long g = (long long)blockIdx.x * 256 + threadIdx.x;
  for (; g + stride < n8; g += 2 * stride) {
    convert(g);
    convert(g + stride);
  }
  if (g < n8) convert(g);
}

// ------------------------------------------------------------ dK/dV kernel
// Work item = one tile of 128 keys (the MMA M dimension for S^T, dP^T, dV, dK)
// of one head, walking the query tiles of BM rows that can see it; one
// persistent CTA per SM runs items back to back.  With DSPLIT = 2 each of two
// items keeps half of the d columns of dV and dK (head dim 256).
//
//   S^T  = K Q^T     (A = K K-major, B = Q K-major)          -> TMEM fp32
//   dP^T = V dO^T    (A = V K-major, B = dO K-major)          -> TMEM fp32
//   P^T  = exp2(S^T*c - lse2), dS^T = P^T o (dP^T - D)       (thread = key row)
//   dV  += P^T dO    (A = P^T from TMEM, B = dO MN-major)
//   dK  += dS^T Q    (A = dS^T from TMEM, B = Q MN-major)
//   5-GEMM, d = 128: dQ^T = K^T dS^T (A = K MN-major, B = dS^T smem MN-major),
//                    lanes = d;  d = 64: dQ = dS K (A = dS^T smem MN-major,
//                    B = K MN-major), lanes = query.  Drained by the last
//                    warpgroup through shared memory into bulk fp32 reductions.
//
// SEP: P^T and dS^T get their own TMEM columns, so S^T(i+1) and dP^T(i+1) are
// issued before dV(i), dK(i), dQ(i) and overlap the softmax of tile i+1.
// Otherwise they alias the S^T / dP^T columns and the MMA order is sequential.
// VT: V lives in TMEM (written by the compute warps, thread = key row) and
// dP^T = V dO^T takes A from TMEM; the 64 KB of shared memory this saves at
// d = 256 holds a second query stage.
// OS (7-GEMM, d = 256): the two work items of a key tile split the outputs
// instead of the columns of d: item h = 0 computes S^T, P^T and dV only (no
// dP^T), item h = 1 computes S^T, dP^T, dS^T and dK; each keeps one 256-column
// accumulator in the same TMEM columns.
struct BwdKVParams {
  CUtensorMap q_map;   // box {64, BM, 1}
  CUtensorMap k_map;   // box {64, 128, 1}
  CUtensorMap v_map;   // box {64, 128, 1}
  CUtensorMap do_map;  // box {64, BM, 1}
  const uint16_t* v;   // bf16 [BH, N, hd] (read row by row into TMEM by VT configurations)
  const float* lse2;
  const float* dd;
  float* dqacc;
  uint16_t* dk;
  uint16_t* dv;
  int* err;
  int N, Npad, BH;
  int hd;  // head dim of the tensors (<= D; tile columns past it read as 0 and are not stored)
  float scale_log2;
  float scale;
  int causal;
  int group;  // heads per launch-order group
  int items;  // work items (key tiles x query parts x d parts x heads); the grid is persistent over them
  int* sched; // next unclaimed work item (zero at launch)
  // Query-range split (few heads, long sequences): each key tile's query tiles are
  // cut into `qsplit` contiguous parts, each a work item of its own.  With
  // qsplit > 1 an item writes its fp32 dK and dV sums over its part (dK without
  // the scale) to dkpart / dvpart [qsplit][BH][Npad][D] instead of dk / dv, and
  // bwd_kvsum_kernel adds the parts.
  int qsplit;
  float* dkpart;
  float* dvpart;
};

// Sum of the query-range parts of dK and dV: dV = sum_s dvpart[s], dK = scale *
// sum_s dkpart[s] (parts in fixed order, so the result is reproducible), bf16.
struct KVSumParams {
  const float* dkpart;
  const float* dvpart;
  uint16_t* dk;
  uint16_t* dv;
  int* err;
  int N, Npad, BH, hd, D, parts;
  float scale;
};

static __global__ void __launch_bounds__(256) bwd_kvsum_kernel(const KVSumParams p) {
  grid_dep_wait();
  if (*reinterpret_cast<volatile const int*>(p.err) != 0) return;
  const int tpr = p.hd / 8;
  const long long g = (long long)blockIdx.x * 256 + threadIdx.x;
  const long long row = g / tpr;  // bh * N + j
  if (row >= (long long)p.BH * p.N) return;
  const int c = (int)(g - row * tpr) * 8;
  const int bh = (int)(row / p.N), j = (int)(row % p.N);
  const size_t off = ((size_t)bh * p.Npad + j) * p.D + c;
  const size_t stride = (size_t)p.BH * p.Npad * p.D;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, b[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < p.parts; ++s) {
    const float4* v4 = reinterpret_cast<const float4*>(p.dvpart + s * stride + off);
    const float4* k4 = reinterpret_cast<const float4*>(p.dkpart + s * stride + off);
    const float4 v0 = v4[0], v1 = v4[1], k0 = k4[0], k1 = k4[1];
    a[0] += v0.x; a[1] += v0.y; a[2] += v0.z; a[3] += v0.w;
    a[4] += v1.x; a[5] += v1.y; a[6] += v1.z; a[7] += v1.w;
    b[0] += k0.x; b[1] += k0.y; b[2] += k0.z; b[3] += k0.w;
    b[4] += k1.x; b[5] += k1.y; b[6] += k1.z; b[7] += k1.w;
  }
  const float sc = p.scale;
  *reinterpret_cast<uint4*>(p.dv + (size_t)row * p.hd + c) =
      make_uint4(pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]), pack_bf16(a[6], a[7]));
  *reinterpret_cast<uint4*>(p.dk + (size_t)row * p.hd + c) =
      make_uint4(pack_bf16(b[0] * sc, b[1] * sc), pack_bf16(b[2] * sc, b[3] * sc), pack_bf16(b[4] * sc, b[5] * sc),
                 pack_bf16(b[6] * sc, b[7] * sc));
}

template <int D_, int BM_, bool DQ_, int DSPLIT_, int QS_, bool SEP_, bool VT_ = false, bool OS_ = false>
struct BwdKVCfg {
  static constexpr int D = D_, BM = BM_, DSPLIT = DSPLIT_, QS = QS_;
  static constexpr bool DQ = DQ_, SEP = SEP_, VT = VT_, OS = OS_;
  // EARLY: the compute warps load all of S^T / dP^T into registers and release
  // those TMEM columns at once, so S^T(i+1), dP^T(i+1) run during the softmax of i.
  static constexpr bool EARLY = SEP && BM == 64;
  // Compute warpgroups: the 5-GEMM kernels (d = 128 with EARLY, and d = 64)
  // split the BM query columns (and the dV / dK epilogue) over two warpgroups to
  // halve the per-tile critical path; the 7-GEMM kernels measured faster with one.
  static constexpr int NCW = (DQ && (EARLY || D == 64)) ? 2 : 1;
  static constexpr int CW = BM / NCW;
  // ALLREG (7-GEMM, P^T / dS^T over S^T / dP^T, 64 query columns): all of a tile's
  // S^T and dP^T columns are loaded with one wait, computed, then stored, instead of
  // a load-wait round trip per 32 columns.
  static constexpr bool ALLREG = !SEP && !EARLY && !DQ && CW == 64;
  // Without separate P^T / dS^T columns, each compute warpgroup packs its results
  // over the first half of its own S^T / dP^T columns (no warpgroup overwrites
  // columns the other still reads).  Packed column of query column c:
  static constexpr bool SPLITPACK = !SEP && NCW == 2;
  static __device__ __forceinline__ int pcol(int c) { return SPLITPACK ? (c / CW) * CW + (c % CW) / 2 : c / 2; }
  static constexpr int DRAIN_W0 = 4 + 4 * NCW;  // first dQ drain warp (5-GEMM)
  static constexpr bool DQ_T = DQ && D == 128;  // dQ^T (lanes = d) vs dQ (lanes = query)
  static constexpr int BN = 128;
  static constexpr int DH = OS ? D : D / DSPLIT;  // accumulator columns per item
  static constexpr int PANELS = D / 64;
  static constexpr uint32_t KV_PANEL = BN * 128;
  static constexpr uint32_t KV_TILE = PANELS * KV_PANEL;
  static constexpr uint32_t QD_PANEL = BM * 128;
  static constexpr uint32_t QD_TILE = PANELS * QD_PANEL;
  static constexpr uint32_t DS_PANEL = BN * 128;  // dS^T smem [128 keys][BM queries]
  static constexpr uint32_t DS_TILE = (BM / 64) * DS_PANEL;
  static constexpr int PREFETCH = QS + 2;  // query tiles ahead for L2 prefetch
  static constexpr uint32_t STAGE_TX = 2 * QD_TILE + 2 * BM * 4;  // bytes landing per stage
  static constexpr uint32_t STAGE_BYTES = (STAGE_TX + 1023) / 1024 * 1024;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + KV_TILE;
  static constexpr uint32_t OFF_STAGE = OFF_V + (VT ? 0 : KV_TILE);  // Q, dO, lse2, dd per stage
  static constexpr uint32_t OFF_DS = OFF_STAGE + QS * STAGE_BYTES;
  static constexpr uint32_t OFF_STG = OFF_DS + (DQ ? DS_TILE : 0);
  // Shared-memory staging for the bulk dQ reductions (one query tile of fp32).
  static constexpr uint32_t STG_BYTES = DQ ? BM * D * 4 : 0;
  static constexpr uint32_t OFF_BAR = OFF_STG + STG_BYTES;
  static constexpr int B_KV = 0, B_QDFULL = 1, B_QDEMPTY = 1 + QS, B_SDP = 1 + 2 * QS,
                       B_PDS = B_SDP + 1, B_MMA = B_PDS + 1, B_DQFULL = B_MMA + 1,
                       B_DQFREE = B_DQFULL + 1, B_STGFREE = B_DQFREE + 1, B_STGFULL = B_STGFREE + 1,
                       B_SCONS = B_STGFULL + 1, B_DONE = B_SCONS + 1, B_KVEMPTY = B_DONE + 1,
                       B_ITEMFULL = B_KVEMPTY + 1, B_ITEMEMPTY = B_ITEMFULL + 4, B_VREADY = B_ITEMEMPTY + 4,
                       NBAR = B_VREADY + 1;
  static constexpr int IQ = 4;  // claimed work items passed from the producer to the other roles
  // Roles that read each work item: the MMA issuing thread(s), the compute warps, the drain warps.
  static constexpr int ITEM_READERS = (EARLY ? 2 : 1) + 4 * NCW + (DQ ? 4 : 0);
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 32 + 1024;
  // TMEM columns
  static constexpr int T_ST = 0, T_DPT = BM;
  static constexpr int T_PT = SEP ? 2 * BM : T_ST;
  static constexpr int T_DST = SEP ? 2 * BM + BM / 2 : T_DPT;
  static constexpr int T_ACC = SEP ? 3 * BM : 2 * BM;
  static constexpr int T_DV = T_ACC, T_DK = T_ACC + (OS ? 0 : DH), T_DQ = T_ACC + (OS ? 1 : 2) * DH;
  static constexpr int DQ_COLS = DQ ? (DQ_T ? BM : D) : 0;
  static constexpr int T_V = T_DQ + DQ_COLS;  // VT: V as packed bf16 pairs, D / 2 columns
  static constexpr int TMEM_USED = T_V + (VT ? D / 2 : 0);
  static constexpr uint32_t TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
  static constexpr int THREADS = 128 * (1 + NCW + (DQ ? 1 : 0));
  // setmaxnreg budgets per warpgroup (producer/MMA, compute, dQ drain): the sum
  // over warpgroups stays within the launch's THREADS * (65536 / THREADS),
  // i.e. 72 + 2 * 160 + 120 = 512 at 512 threads and 104 + 224 + 168 <= 3 * 168.
  static constexpr int REG_LAUNCH = 65536 / THREADS >= 256 ? 255 : (65536 / THREADS) / 8 * 8;
  static constexpr int REG_LOW = THREADS == 512 ? 72 : 104;
  static constexpr int REG_COMPUTE = THREADS == 512 ? 160 : (NCW == 2 ? 208 : 224);
  static constexpr int REG_DRAIN = THREADS == 512 ? 120 : REG_LAUNCH;
  static_assert(THREADS < 384 || REG_LOW + NCW * REG_COMPUTE + (DQ ? REG_DRAIN : 0) <= THREADS / 128 * REG_LAUNCH,
                "register split exceeds the launch budget");
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(!SEP || QS >= 2, "overlapped order needs two query stages");
  static_assert(!DQ || DSPLIT == 1, "5-GEMM keeps all of dQ's columns");
  static_assert(!DQ || D == 64 ? true : (D == 128 && BM == 64), "dQ^T path needs M = d = 128");
  static_assert(!(DQ && D == 64) || BM == 128, "dQ path needs M = BM = 128");
  static_assert(!VT || (!EARLY && NCW == 1), "V in TMEM is written by the single compute warpgroup");
  static_assert(!OS || (VT && !DQ && !SEP && DSPLIT == 2), "output split: dV item and dK item per key tile");
};

// FEW: the instantiation for launches with few work items (fewer than about four
// per SM: few heads), with the query-range split (p.qsplit >= 1) and each item's
// query-tile walk starting at its own offset; the plain one keeps one part per
// key tile and the natural order as constants and has no partial-sum epilogue.
template <class C, bool FEW>
__global__ void __launch_bounds__(C::THREADS, 1) bwd_kv_kernel(const __grid_constant__ BwdKVParams p) {
  constexpr int D = C::D, BM = C::BM, QS = C::QS, DH = C::DH;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw_addr);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 4);
  // Query tiles whose dV / dK / dQ MMAs have been issued (EARLY issue order).
  volatile int* tails_issued = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 12);
  const int warp = warp_id();
  const int lane = lane_id();
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *tails_issued = 0;
    mbar_init(BAR(C::B_KV), 1);
    mbar_init(BAR(C::B_KVEMPTY), C::EARLY ? 2 : 1);
    for (int k = 0; k < C::IQ; ++k) {
      mbar_init(BAR(C::B_ITEMFULL + k), 1);
      mbar_init(BAR(C::B_ITEMEMPTY + k), C::ITEM_READERS);
    }
    for (int s = 0; s < QS; ++s) {
      mbar_init(BAR(C::B_QDFULL + s), 1);
      mbar_init(BAR(C::B_QDEMPTY + s), 1);
    }
    mbar_init(BAR(C::B_SDP), 1);
    mbar_init(BAR(C::B_PDS), 4 * C::NCW);
    mbar_init(BAR(C::B_MMA), 1);
    mbar_init(BAR(C::B_DQFULL), 1);
    mbar_init(BAR(C::B_DQFREE), 4);
    mbar_init(BAR(C::B_STGFREE), 1);
    mbar_init(BAR(C::B_STGFULL), 4);
    mbar_init(BAR(C::B_SCONS), 4 * C::NCW);
    mbar_init(BAR(C::B_DONE), C::EARLY ? 2 : 1);
    mbar_init(BAR(C::B_VREADY), 4 * C::NCW);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const CtaAbort ab{abort_flag, p.err};
  grid_dep_wait();
  // A kernel that gave up earlier left the error word set: do nothing.
  const bool skip = *reinterpret_cast<volatile int*>(p.err) != 0;

  // Persistent work loop.  Work item w = (key tile, d part, head) in launch
  // order: heads in groups for L2 reuse of their Q, dO and dQ accumulator,
  // and inside a group the key tiles that the most query tiles see first
  // (under the causal mask), heads varying fastest.  The producer claims items
  // from a global counter one item ahead (so idle SMs take the next item,
  // longest first) and passes each claimed index through a small shared-memory
  // ring to the other roles.  Every role walks the same items and counts the
  // same query tiles, so barrier phases run on across items.
  const int n_kt = (p.N + C::BN - 1) / C::BN;
  const int n_qt = (p.N + BM - 1) / BM;
  volatile int* item_ring = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 16);
  // Item claimed t-th by this CTA (>= p.items once the counter ran out), or -1
  // if the wait gave up.  Single-thread readers.
  auto item_one = [&](int t) -> int {
    const int k = t % C::IQ;
    if (!wait_one(BAR(C::B_ITEMFULL + k), (t / C::IQ) & 1, ab, (kKBwdKV << 8) | 18)) return -1;
    const int w = item_ring[k];
    mbar_arrive(BAR(C::B_ITEMEMPTY + k));
    return w;
  };
  // The same for a whole warp (lane 0 releases the slot).
  auto item_warp = [&](int t) -> int {
    const int k = t % C::IQ;
    if (!wait_warp(BAR(C::B_ITEMFULL + k), (t / C::IQ) & 1, ab, (kKBwdKV << 8) | 18)) return -1;
    const int w = item_ring[k];
    __syncwarp();
    if (lane_id() == 0) mbar_arrive(BAR(C::B_ITEMEMPTY + k));
    return w;
  };
  struct Item {
    int bh, h, part, k0, qt0, n;  // head, d part, query part, first key, first query tile, query tiles
    int rot;                      // the item's first step takes query tile qt0 + rot (see qt_at)
  };
  // Item w: key tile, query part and d part from the launch order; the key tile's
  // query tiles (from the diagonal under the causal mask) are cut into p.qsplit
  // contiguous parts (some possibly empty when there are fewer tiles than parts).
  const int qsplit = FEW ? p.qsplit : 1;
  auto coords = [&](int w) {
    Item I;
    int tile;
    grouped_order(w, n_kt * C::DSPLIT * qsplit, p.BH, p.group, tile, I.bh);
    I.h = tile % C::DSPLIT;
    const int kq = tile / C::DSPLIT;
    if constexpr (FEW) {
      I.part = kq % qsplit;
      I.k0 = (kq / qsplit) * C::BN;
      const int first = p.causal ? I.k0 / BM : 0;
      const int total = n_qt - first;
      I.qt0 = first + (int)((long long)I.part * total / qsplit);
      I.n = first + (int)((long long)(I.part + 1) * total / qsplit) - I.qt0;
    } else {
      I.part = 0;
      I.k0 = kq * C::BN;
      I.qt0 = p.causal ? I.k0 / BM : 0;
      I.n = n_qt - I.qt0;
    }
    // With few heads, items of one head that run at the same time would otherwise
    // walk the same query tiles in step (all of them from the first tile without
    // the mask) and reduce into the same dQ rows at once; each key tile starts its
    // walk at its own offset (n * kt / n_kt) and wraps around (measured +2 to +6 %
    // with one to eight heads, -2.5 % with 64 heads of 2048 rows, where concurrent
    // items belong to different heads anyway).
    I.rot = (FEW && I.n > 0) ? (int)((long long)I.n * (I.k0 / C::BN) / n_kt) : 0;
    return I;
  };
  // Query tile of step i of item I.
  auto qt_at = [](const Item& I, int i) {
    const int j = i + I.rot;
    return I.qt0 + (j >= I.n ? j - I.n : j);
  };

  auto stage_q = [&](int s) { return sbase + C::OFF_STAGE + s * C::STAGE_BYTES; };
  auto stage_do = [&](int s) { return stage_q(s) + C::QD_TILE; };
  auto stage_lse = [&](int s) { return stage_q(s) + 2 * C::QD_TILE; };
  auto stage_dd = [&](int s) { return stage_lse(s) + BM * 4; };

  // With 384 or 512 threads each role branch starts with its warpgroup's
  // register budget (REG_LOW, REG_COMPUTE, REG_DRAIN): the producer/MMA
  // warpgroup gives registers to the compute warpgroup(s).
  constexpr bool kSplitRegs = C::THREADS >= 384;
  if (!skip) {
    if (warp < 4) {
    if constexpr (kSplitRegs) regs_shrink<C::REG_LOW>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      // Query-tile stages run on across items.  An item's first stages are
      // issued before its K/V tile, which has to wait until the previous
      // item's last MMAs have read K and V.
      if (lane == 0) {
        tma_prefetch_desc(&p.q_map);
        tma_prefetch_desc(&p.k_map);
        tma_prefetch_desc(&p.v_map);
        tma_prefetch_desc(&p.do_map);
        int it = 0, nkv = 0;
        bool ok = true;
        auto prefetch_qd = [&](const Item& I, int i) {
          const int prow = qt_at(I, i) * BM;
          for (int pn = 0; pn < C::PANELS; ++pn) {
            tma_prefetch_l2_3d(&p.q_map, 64 * pn, prow, I.bh);
            tma_prefetch_l2_3d(&p.do_map, 64 * pn, prow, I.bh);
          }
        };
        int published = 0;
        auto publish = [&](int w) -> bool {
          const int k = published % C::IQ;
          if (!wait_one(BAR(C::B_ITEMEMPTY + k), ((published / C::IQ) & 1) ^ 1, ab, (kKBwdKV << 8) | 17))
            return false;
          item_ring[k] = w;
          mbar_arrive(BAR(C::B_ITEMFULL + k));
          ++published;
          return true;
        };
        // 5-GEMM: the first item of CTA c is item c (the grid never exceeds the
        // items) and the counter hands out the rest, so no CTA starts behind a
        // contended atomic (measured -1 % on 64 heads of 2048 rows, -4 % on one
        // head of 16384; the 7-GEMM kernels measured 1 % slower with it at d = 256
        // and claim every item).
        const int first = C::DQ ? (int)gridDim.x : 0;
        int wn = C::DQ ? (int)blockIdx.x : atomicAdd(p.sched, 1);
        ok = publish(wn);
        while (ok && wn < p.items) {
          const int w = wn;
          wn = first + atomicAdd(p.sched, 1);
          if (!publish(wn)) break;
          const Item I = coords(w);
          if (I.n <= 0) continue;
          const bool has_next = wn < p.items;
          const Item J = has_next ? coords(wn) : I;
          auto issue_stage = [&](int i) -> bool {
            const int s = it % QS;
            if (!wait_one(BAR(C::B_QDEMPTY + s), ((it / QS) & 1) ^ 1, ab, (kKBwdKV << 8) | 1)) return false;
            const int qrow = qt_at(I, i) * BM;
            mbar_expect_tx(BAR(C::B_QDFULL + s), C::STAGE_TX);
            for (int pn = 0; pn < C::PANELS; ++pn) {
              tma_load_3d(stage_q(s) + pn * C::QD_PANEL, &p.q_map, BAR(C::B_QDFULL + s), 64 * pn, qrow, I.bh);
              tma_load_3d(stage_do(s) + pn * C::QD_PANEL, &p.do_map, BAR(C::B_QDFULL + s), 64 * pn, qrow, I.bh);
            }
            bulk_load(stage_lse(s), p.lse2 + (size_t)I.bh * p.Npad + qrow, BM * 4, BAR(C::B_QDFULL + s));
            bulk_load(stage_dd(s), p.dd + (size_t)I.bh * p.Npad + qrow, BM * 4, BAR(C::B_QDFULL + s));
            ++it;
            // Stage loads can only start once a slot frees up (a few tiles ahead of
            // use); pull the tiles further ahead, into the next item, into L2.
            const int ahead = i + C::PREFETCH;
            if (ahead < I.n) prefetch_qd(I, ahead);
            else if (has_next && ahead - I.n < J.n) prefetch_qd(J, ahead - I.n);
            return true;
          };
          const int pre = min(QS - 1, I.n);
          int i = 0;
          for (; ok && i < pre; ++i) ok = issue_stage(i);
          if (!ok) break;
          if (nkv > 0 && !wait_one(BAR(C::B_KVEMPTY), (nkv - 1) & 1, ab, (kKBwdKV << 8) | 15)) break;
          mbar_expect_tx(BAR(C::B_KV), (C::VT ? 1 : 2) * C::KV_TILE);
          for (int pn = 0; pn < C::PANELS; ++pn) {
            tma_load_3d(sbase + C::OFF_K + pn * C::KV_PANEL, &p.k_map, BAR(C::B_KV), 64 * pn, I.k0, I.bh);
            if (!C::VT)
              tma_load_3d(sbase + C::OFF_V + pn * C::KV_PANEL, &p.v_map, BAR(C::B_KV), 64 * pn, I.k0, I.bh);
          }
          ++nkv;
          if (has_next)
            for (int pn = 0; pn < C::PANELS; ++pn) {
              tma_prefetch_l2_3d(&p.k_map, 64 * pn, J.k0, J.bh);
              tma_prefetch_l2_3d(&p.v_map, 64 * pn, J.k0, J.bh);
            }
          for (; ok && i < I.n; ++i) ok = issue_stage(i);
        }
        if (nkv > 0) wait_drain_bwd(BAR(C::B_KV), (nkv - 1) & 1);
        for (int j = max(0, it - QS); j < it; ++j) wait_drain_bwd(BAR(C::B_QDFULL + j % QS), (j / QS) & 1);
      }
      __syncwarp();
    } else if (warp == 1 || (C::EARLY && warp == 2)) {
      // ---------------------------------------------------------- MMA issue
      // EARLY configurations use two issuing threads: warp 1 issues S^T / dP^T,
      // warp 2 issues dV, dK and dQ.  The two streams touch disjoint TMEM columns
      // and are ordered only through the compute warps' barriers, so a thread
      // blocked on a commit or a wait no longer leaves the tensor pipe idle.
      // Each issuing thread commits to KVEMPTY after its last MMA of an item
      // that reads K or V.  The tensor pipe runs MMAs in issue order and the
      // compute warps need dV/dK/dQ(g-2) done before they store P^T / dS^T(g-1),
      // so S^T(g) is issued only after dV/dK/dQ(g-2) (measured +3..11 %).
      {
        constexpr uint32_t idS = make_idesc(128, BM, false, false);
        constexpr uint32_t idAcc = make_idesc(128, DH, false, true);
        const uint32_t kt = sbase + C::OFF_K, vt = sbase + C::OFF_V;
        auto issue_s = [&](int s) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss(tmem + C::T_ST, desc_kmajor(kt, C::KV_PANEL, 16 * k),
                   desc_kmajor(stage_q(s), C::QD_PANEL, 16 * k), idS, k > 0 ? 1u : 0u);
        };
        auto issue_dp = [&](int s) {
          if constexpr (C::VT) {
            // A = V from TMEM: 16 keys' worth of d per MMA is 8 packed columns.
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_ts(tmem + C::T_DPT, tmem + C::T_V + 8 * k, desc_kmajor(stage_do(s), C::QD_PANEL, 16 * k), idS,
                     k > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_ss(tmem + C::T_DPT, desc_kmajor(vt, C::KV_PANEL, 16 * k),
                     desc_kmajor(stage_do(s), C::QD_PANEL, 16 * k), idS, k > 0 ? 1u : 0u);
          }
          mma_commit(BAR(C::B_SDP));
        };
        auto issue_sdp = [&](int s) {
          issue_s(s);
          issue_dp(s);
        };
        auto issue_acc = [&](int s, int h, bool first) {
          const int hoff = C::OS ? 0 : h;  // d part of the accumulators
          const uint32_t dob = stage_do(s) + hoff * (DH / 64) * C::QD_PANEL;
          const uint32_t qb = stage_q(s) + hoff * (DH / 64) * C::QD_PANEL;
          if (!C::OS || h == 0) {
#pragma unroll
            for (int k = 0; k < BM / 16; ++k)
              mma_ts(tmem + C::T_DV, tmem + C::T_PT + C::pcol(16 * k), desc_mnmajor(dob, C::QD_PANEL, 16 * k), idAcc,
                     (!first || k > 0) ? 1u : 0u);
          }
          if (!C::OS || h == 1) {
#pragma unroll
            for (int k = 0; k < BM / 16; ++k)
              mma_ts(tmem + C::T_DK, tmem + C::T_DST + C::pcol(16 * k), desc_mnmajor(qb, C::QD_PANEL, 16 * k), idAcc,
                     (!first || k > 0) ? 1u : 0u);
          }
        };
        // OS: the dV item needs no dP^T.
        auto issue_sdp_h = [&](int s, int h) {
          issue_s(s);
          if (C::OS && h == 0)
            mma_commit(BAR(C::B_SDP));
          else
            issue_dp(s);
        };
        auto issue_dq = [&]() {
          const uint32_t ds = sbase + C::OFF_DS;
          if constexpr (C::DQ_T) {
            constexpr uint32_t id = make_idesc(128, BM, true, true);
#pragma unroll
            for (int k = 0; k < C::BN / 16; ++k)
              mma_ss(tmem + C::T_DQ, desc_mnmajor(kt, C::KV_PANEL, 16 * k), desc_mnmajor(ds, C::DS_PANEL, 16 * k),
                     id, k > 0 ? 1u : 0u);
          } else {
            constexpr uint32_t id = make_idesc(128, D, true, true);
#pragma unroll
            for (int k = 0; k < C::BN / 16; ++k)
              mma_ss(tmem + C::T_DQ, desc_mnmajor(ds, C::DS_PANEL, 16 * k), desc_mnmajor(kt, C::KV_PANEL, 16 * k),
                     id, k > 0 ? 1u : 0u);
          }
          mma_commit(BAR(C::B_DQFULL));
        };
        // dV, dK (and dQ) of query tile g (stage s), then the commits that free
        // the stage and tell the compute warps P^T / dS^T have been read.
        auto issue_tail = [&](int g, int s, int h, bool first) -> bool {
          issue_acc(s, h, first);
          if constexpr (C::DQ) {
            if (g > 0 && !wait_warp(BAR(C::B_DQFREE), (g - 1) & 1, ab, (kKBwdKV << 8) | 6)) return false;
            tc_fence_after();
            issue_dq();
          }
          mma_commit(BAR(C::B_MMA));
          mma_commit(BAR(C::B_QDEMPTY + s));
          return true;
        };
        bool ok = true;
        int g = 0, nkv = 0;
        if (C::EARLY && warp == 1) {
          // S^T(g), dP^T(g) as soon as the compute warps hold S^T(g-1), dP^T(g-1) in registers.
          for (int r = 0; ok; ++r) {
            const int w = item_warp(r);
            if (w < 0 || w >= p.items) break;
            const int n = coords(w).n;
            if (n <= 0) continue;
            if (!wait_warp(BAR(C::B_KV), nkv & 1, ab, (kKBwdKV << 8) | 2)) break;
            for (int i = 0; i < n; ++i, ++g) {
              const int s = g % QS;
              if ((g > 0 && !wait_warp(BAR(C::B_SCONS), (g - 1) & 1, ab, (kKBwdKV << 8) | 14)) ||
                  !__all_sync(0xffffffffu, wait_count(tails_issued, g - 1, ab, (kKBwdKV << 8) | 16)) ||
                  !wait_warp(BAR(C::B_QDFULL + s), (g / QS) & 1, ab, (kKBwdKV << 8) | 5)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_sdp(s);
            }
            if (!ok) break;
            mma_commit(BAR(C::B_KVEMPTY));
            ++nkv;
          }
        } else if (C::EARLY) {
          for (int r = 0; ok; ++r) {
            const int w = item_warp(r);
            if (w < 0 || w >= p.items) break;
            const Item I = coords(w);
            if (I.n <= 0) continue;
            for (int i = 0; i < I.n; ++i, ++g) {
              const int s = g % QS;
              if (!wait_warp(BAR(C::B_PDS), g & 1, ab, (kKBwdKV << 8) | 4)) {
                ok = false;
                break;
              }
              tc_fence_after();
              if (!issue_tail(g, s, I.h, i == 0)) {
                ok = false;
                break;
              }
              *tails_issued = g + 1;
            }
            if (!ok) break;
            mma_commit(BAR(C::B_KVEMPTY));
          }
        } else {
          int nv = 0;  // items whose V the compute warps wrote into TMEM (VT)
          for (int r = 0; ok; ++r) {
            const int w = item_warp(r);
            if (w < 0 || w >= p.items) break;
            const Item I = coords(w);
            if (I.n <= 0) continue;
            if (!wait_warp(BAR(C::B_KV), nkv & 1, ab, (kKBwdKV << 8) | 2) ||
                !wait_warp(BAR(C::B_QDFULL + g % QS), (g / QS) & 1, ab, (kKBwdKV << 8) | 3))
              break;
            tc_fence_after();
            issue_s(g % QS);
            if (C::OS && I.h == 0) {
              mma_commit(BAR(C::B_SDP));
            } else {
              // VT: the compute warps have written this item's V into TMEM.
              if (C::VT && !wait_warp(BAR(C::B_VREADY), nv & 1, ab, (kKBwdKV << 8) | 19)) break;
              if (C::VT) ++nv;
              tc_fence_after();
              issue_dp(g % QS);
            }
            for (int i = 0; i < I.n; ++i, ++g) {
              const int s = g % QS;
              const int s1 = (g + 1) % QS;
              if (!wait_warp(BAR(C::B_PDS), g & 1, ab, (kKBwdKV << 8) | 4)) {
                ok = false;
                break;
              }
              tc_fence_after();
              // SEP: S^T / dP^T of the next query tile go ahead of dV, dK, dQ.
              if (C::SEP && i + 1 < I.n) {
                if (!wait_warp(BAR(C::B_QDFULL + s1), ((g + 1) / QS) & 1, ab, (kKBwdKV << 8) | 5)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                issue_sdp_h(s1, I.h);
              }
              if (!issue_tail(g, s, I.h, i == 0)) {
                ok = false;
                break;
              }
              if (!C::SEP && i + 1 < I.n) {
                if (!wait_warp(BAR(C::B_QDFULL + s1), ((g + 1) / QS) & 1, ab, (kKBwdKV << 8) | 5)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                issue_sdp_h(s1, I.h);
              }
            }
            if (!ok) break;
            mma_commit(BAR(C::B_KVEMPTY));
            ++nkv;
          }
        }
        mma_commit(BAR(C::B_DONE));
        wait_drain_bwd(BAR(C::B_DONE), 0);
      }
      __syncwarp();
    }
    } else if (warp < C::DRAIN_W0) {
      // ---------------------------------------------- P^T / dS^T (thread = key row)
      if constexpr (kSplitRegs) regs_grow<C::REG_COMPUTE>();
      const int cw = (warp - 4) >> 2;      // compute warpgroup: query columns [c_lo, c_lo + CW)
      const int c_lo = cw * C::CW;
      const int quad = warp & 3;
      const int r = quad * 32 + lane;
      const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
      const float cs = p.scale_log2;
      uint8_t* ds_row = gbase + C::OFF_DS + r * 128;
      bool ok = true;
      int g = 0;
      for (int rr = 0; ok; ++rr) {
        const int w = item_warp(rr);
        if (w < 0 || w >= p.items) break;
        const Item I = coords(w);
        const int kj = I.k0 + r;
        const bool key_ok = kj < p.N;
        if (I.n <= 0) {
          // No query of this item can see the key tile: zero gradients (zero partial
          // sums under the query-range split).
          const int c_off = C::OS ? 0 : I.h * DH;
          if (FEW && p.qsplit > 1) {
            if (key_ok && cw == 0) {
              const size_t off = (((size_t)I.part * p.BH + I.bh) * p.Npad + kj) * D + c_off;
              for (int c = 0; c < DH; c += 4) {
                if (!C::OS || I.h == 0) *reinterpret_cast<float4*>(p.dvpart + off + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                if (!C::OS || I.h == 1) *reinterpret_cast<float4*>(p.dkpart + off + c) = make_float4(0.f, 0.f, 0.f, 0.f);
              }
            }
            continue;
          }
          if (key_ok && cw == 0)
            for (int c = 0; c < DH; c += 8) {
              if (c_off + c < p.hd) {
                if (!C::OS || I.h == 0)
                  *reinterpret_cast<uint4*>(p.dv + ((size_t)I.bh * p.N + kj) * p.hd + c_off + c) = make_uint4(0, 0, 0, 0);
                if (!C::OS || I.h == 1)
                  *reinterpret_cast<uint4*>(p.dk + ((size_t)I.bh * p.N + kj) * p.hd + c_off + c) = make_uint4(0, 0, 0, 0);
              }
            }
          continue;
        }
        if (C::VT && (!C::OS || I.h == 1)) {
          // This item's V row kj as packed bf16 pairs into TMEM lane r: the A
          // operand of dP^T = V dO^T.  The previous item's dP^T MMAs, the last
          // readers of these columns, completed before its last S^T / dP^T
          // barrier, which these warps have waited on.
          const uint16_t* vrow = p.v + ((size_t)I.bh * p.N + (key_ok ? kj : 0)) * p.hd;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 64) {
            uint32_t vw[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              uint4 x = make_uint4(0u, 0u, 0u, 0u);
              if (key_ok && c0 + 8 * u < p.hd) x = *reinterpret_cast<const uint4*>(vrow + c0 + 8 * u);
              vw[4 * u] = x.x;
              vw[4 * u + 1] = x.y;
              vw[4 * u + 2] = x.z;
              vw[4 * u + 3] = x.w;
            }
            tmem_st_32x32b_x32(trow + C::T_V + (c0 >> 1), vw);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C::B_VREADY));
        }
        for (int i = 0; i < I.n; ++i, ++g) {
          const int s = g % QS;
          const int q0 = qt_at(I, i) * BM;
          if (!wait_warp(BAR(C::B_SDP), g & 1, ab, (kKBwdKV << 8) | 7) ||
              !wait_warp(BAR(C::B_QDFULL + s), (g / QS) & 1, ab, (kKBwdKV << 8) | 8)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float* L = reinterpret_cast<const float*>(gbase + (stage_lse(s) - sbase));
          const float* Dd = reinterpret_cast<const float*>(gbase + (stage_dd(s) - sbase));
          const int lim = p.causal ? kj - q0 : -1;  // columns c < lim are masked (query < key)
          // Writes one 32-column chunk of P^T and dS^T (packed bf16) to TMEM and,
          // for the 5-GEMM variant, dS^T row r into the [128 keys][BM queries]
          // swizzled shared-memory tile read by the dQ MMA.
          auto store_chunk = [&](int c0, const uint32_t* pp, const uint32_t* pd) {
            tmem_st_32x32b_x16(trow + C::T_PT + C::pcol(c0), pp);
            tmem_st_32x32b_x16(trow + C::T_DST + C::pcol(c0), pd);
            if constexpr (C::DQ) {
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int ch = (c0 >> 3) + u;
                const int pn = ch >> 3, cc = ch & 7;
                *reinterpret_cast<uint4*>(ds_row + pn * C::DS_PANEL + ((cc ^ (r & 7)) << 4)) =
                    make_uint4(pd[4 * u], pd[4 * u + 1], pd[4 * u + 2], pd[4 * u + 3]);
              }
            }
          };
          constexpr int HOLD = (C::SEP || C::ALLREG) ? C::CW / 2 : 16;
          uint32_t pk_p[HOLD], pk_ds[HOLD];
          // P^T = exp2(S^T c - lse2), dS^T = P^T (dP^T - D) for columns [c0, c0 + 32).
          const float2 c2 = make_float2(cs, cs);
          auto compute_chunk = [&](int c0, const uint32_t* sr, const uint32_t* dr, int hb) {
            // Masks only in chunks that reach past the last key or below the diagonal.
            const bool masked = !key_ok || lim > c0;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 l4 = *reinterpret_cast<const float4*>(L + c0 + e);
              const float4 d4 = *reinterpret_cast<const float4*>(Dd + c0 + e);
              const float2 x01 = ffma2(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2,
                                       make_float2(l4.x, l4.y));
              const float2 x23 = ffma2(make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), c2,
                                       make_float2(l4.z, l4.w));
              float2 p01 = make_float2(ex2(x01.x), ex2(x01.y));
              float2 p23 = make_float2(ex2(x23.x), ex2(x23.y));
              if (masked) {
                const int c = c0 + e;
                if (!key_ok || c < lim) p01.x = 0.f;
                if (!key_ok || c + 1 < lim) p01.y = 0.f;
                if (!key_ok || c + 2 < lim) p23.x = 0.f;
                if (!key_ok || c + 3 < lim) p23.y = 0.f;
              }
              const float2 d01 = fmul2(p01, fadd2(make_float2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])),
                                                  make_float2(d4.x, d4.y)));
              const float2 d23 = fmul2(p23, fadd2(make_float2(__uint_as_float(dr[e + 2]), __uint_as_float(dr[e + 3])),
                                                  make_float2(d4.z, d4.w)));
              pk_p[hb + (e >> 1)] = pack_bf16(p01.x, p01.y);
              pk_p[hb + (e >> 1) + 1] = pack_bf16(p23.x, p23.y);
              pk_ds[hb + (e >> 1)] = pack_bf16(d01.x, d01.y);
              pk_ds[hb + (e >> 1) + 1] = pack_bf16(d23.x, d23.y);
            }
          };
          if constexpr (C::EARLY) {
            uint32_t sr[C::CW], dr[C::CW];
#pragma unroll
            for (int c0 = 0; c0 < C::CW; c0 += 32) {
              tmem_ld_32x32b_x32(trow + C::T_ST + c_lo + c0, sr + c0);
              tmem_ld_32x32b_x32(trow + C::T_DPT + c_lo + c0, dr + c0);
            }
            tmem_wait_ld();
            reg_fence<C::CW>(sr);
            reg_fence<C::CW>(dr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::B_SCONS));
#pragma unroll
            for (int c0 = 0; c0 < C::CW; c0 += 32) compute_chunk(c_lo + c0, sr + c0, dr + c0, c0 >> 1);
          } else if constexpr (C::ALLREG) {
            uint32_t sr[C::CW], dr[C::CW];
#pragma unroll
            for (int c0 = 0; c0 < C::CW; c0 += 32) {
              tmem_ld_32x32b_x32(trow + C::T_ST + c_lo + c0, sr + c0);
              tmem_ld_32x32b_x32(trow + C::T_DPT + c_lo + c0, dr + c0);
            }
            tmem_wait_ld();
            reg_fence<C::CW>(sr);
            reg_fence<C::CW>(dr);
#pragma unroll
            for (int c0 = 0; c0 < C::CW; c0 += 32) compute_chunk(c_lo + c0, sr + c0, dr + c0, c0 >> 1);
#pragma unroll
            for (int c0 = 0; c0 < C::CW; c0 += 32) store_chunk(c_lo + c0, pk_p + (c0 >> 1), pk_ds + (c0 >> 1));
          } else {
#pragma unroll
            for (int c0 = c_lo; c0 < c_lo + C::CW; c0 += 32) {
              uint32_t sr[32], dr[32];
              tmem_ld_32x32b_x32(trow + C::T_ST + c0, sr);
              tmem_ld_32x32b_x32(trow + C::T_DPT + c0, dr);
              tmem_wait_ld();
              reg_fence<32>(sr);
              reg_fence<32>(dr);
              compute_chunk(c0, sr, dr, C::SEP ? ((c0 - c_lo) >> 1) : 0);
              if constexpr (!C::SEP) store_chunk(c0, pk_p, pk_ds);
            }
          }
          if constexpr (C::SEP) {
            // dV, dK, dQ of the previous query tile read P^T, dS^T (TMEM) and dS^T (smem): wait for them.
            if (g > 0 && !wait_warp(BAR(C::B_MMA), (g - 1) & 1, ab, (kKBwdKV << 8) | 9)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < C::CW; c0 += 32) store_chunk(c_lo + c0, pk_p + (c0 >> 1), pk_ds + (c0 >> 1));
          }
          if constexpr (C::DQ) fence_proxy_async_smem();
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C::B_PDS));
        }
        if (!ok) break;
        // ------------------------------------------------ dV, dK epilogue
        // The TMEM reads finish before these warps arrive on PDS for the next
        // item's first query tile, whose dV / dK MMAs overwrite the accumulators.
        if (!wait_warp(BAR(C::B_MMA), (g - 1) & 1, ab, (kKBwdKV << 8) | 10)) break;
        tc_fence_after();
        if (FEW && p.qsplit > 1) {
          // Query-range split: this part's fp32 sums (dK without the scale), one row per thread.
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            if (C::NCW == 2 && which != cw) continue;
            if (C::OS && which != I.h) continue;
            const int c_off = C::OS ? 0 : I.h * DH;
            float* dst = (which == 0 ? p.dvpart : p.dkpart) + (((size_t)I.part * p.BH + I.bh) * p.Npad + kj) * D + c_off;
            const uint32_t tacc = trow + (which == 0 ? C::T_DV : C::T_DK);
#pragma unroll
            for (int c0 = 0; c0 < DH; c0 += 32) {
              uint32_t rv[32];
              tmem_ld_32x32b_x32(tacc + c0, rv);
              tmem_wait_ld();
              reg_fence<32>(rv);
              if (key_ok) {
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                  *reinterpret_cast<float4*>(dst + c0 + e) =
                      make_float4(__uint_as_float(rv[e]), __uint_as_float(rv[e + 1]), __uint_as_float(rv[e + 2]),
                                  __uint_as_float(rv[e + 3]));
              }
            }
          }
          tc_fence_before();
          continue;
        }
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          if (C::NCW == 2 && which != cw) continue;  // two warpgroups: one stores dV, the other dK
          if (C::OS && which != I.h) continue;       // output split: this item's one accumulator
          const int c_off = C::OS ? 0 : I.h * DH;    // first column of this item's d part
          uint16_t* dst = (which == 0 ? p.dv : p.dk) + (size_t)I.bh * p.N * p.hd + c_off;
          const int cols = min(DH, p.hd - c_off);  // stored columns of this d part
          const float mul = which == 0 ? 1.f : p.scale;
          const uint32_t tacc = trow + (which == 0 ? C::T_DV : C::T_DK);
          if constexpr (C::DQ) {
            // Staged through this warp's own footprint of the dS^T tile (free once
            // the last dQ MMA has read it): each thread writes its row, then the warp
            // writes R consecutive 16-byte chunks of 32 / R rows per instruction, so a
            // warp store covers a few contiguous row segments instead of 32 rows.
            constexpr int EW = C::CW < DH ? C::CW : DH;  // columns per round
            constexpr int R = EW / 8;                    // 16-byte chunks per row per round
            static_assert(EW % 32 == 0 && 32 % R == 0, "epilogue staging shape");
            auto ds_chunk = [&](int rr, int u) -> uint4* {
              const int ch = (c_lo >> 3) + u;
              return reinterpret_cast<uint4*>(gbase + C::OFF_DS + (ch >> 3) * C::DS_PANEL + rr * 128 +
                                              (((ch & 7) ^ (rr & 7)) << 4));
            };
#pragma unroll
            for (int c0 = 0; c0 < DH; c0 += EW) {
              uint32_t pk[EW / 2];
#pragma unroll
              for (int cc = 0; cc < EW; cc += 32) {
                uint32_t rv[32];
                tmem_ld_32x32b_x32(tacc + c0 + cc, rv);
                tmem_wait_ld();
                reg_fence<32>(rv);
#pragma unroll
                for (int e = 0; e < 32; e += 2)
                  pk[(cc + e) >> 1] = pack_bf16(__uint_as_float(rv[e]) * mul, __uint_as_float(rv[e + 1]) * mul);
              }
#pragma unroll
              for (int u = 0; u < R; ++u) *ds_chunk(r, u) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
              __syncwarp();
#pragma unroll
              for (int j = 0; j < R; ++j) {
                const int rr = quad * 32 + j * (32 / R) + lane / R;
                const int u = lane % R;
                const uint4 val = *ds_chunk(rr, u);
                if (I.k0 + rr < p.N && c0 + 8 * u < cols)
                  *reinterpret_cast<uint4*>(dst + (size_t)(I.k0 + rr) * p.hd + c0 + 8 * u) = val;
              }
              __syncwarp();
            }
          } else {
            uint16_t* drow = dst + (size_t)(key_ok ? kj : 0) * p.hd;
#pragma unroll
            for (int c0 = 0; c0 < DH; c0 += 32) {
              uint32_t rv[32];
              tmem_ld_32x32b_x32(tacc + c0, rv);
              tmem_wait_ld();
              reg_fence<32>(rv);
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 32; e += 2)
                pk[e >> 1] = pack_bf16(__uint_as_float(rv[e]) * mul, __uint_as_float(rv[e + 1]) * mul);
              if (key_ok) {
                uint4* o4 = reinterpret_cast<uint4*>(drow + c0);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                  if (c0 + 8 * v < cols) o4[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
              }
            }
          }
        }
        tc_fence_before();
      }
    } else {
      if constexpr (C::DQ) {
      // ------------------------------------------------------ dQ drain (5-GEMM)
      if constexpr (kSplitRegs && C::REG_DRAIN < C::REG_LAUNCH) regs_shrink<C::REG_DRAIN>();
      const int quad = warp & 3;
      const int lr = quad * 32 + lane;  // TMEM lane: d index (dQ^T) or query row (dQ)
      const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16) + C::T_DQ;
      float* stg = reinterpret_cast<float*>(gbase + C::OFF_STG);
      const bool leader = (warp == C::DRAIN_W0 && lane == 0);
      bool ok = true;
      int g = 0;
      for (int rr = 0; ok; ++rr) {
        const int w = item_warp(rr);
        if (w < 0 || w >= p.items) break;
        const Item I = coords(w);
        for (int i = 0; i < I.n; ++i, ++g) {
          if (!wait_warp(BAR(C::B_DQFULL), g & 1, ab, (kKBwdKV << 8) | 11)) {
            ok = false;
            break;
          }
          tc_fence_after();
          constexpr int COLS = C::DQ_COLS;
          uint32_t v[COLS];
#pragma unroll
          for (int c0 = 0; c0 < COLS; c0 += 32) tmem_ld_32x32b_x32(trow + c0, v + c0);
          tmem_wait_ld();
          reg_fence<COLS>(v);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C::B_DQFREE));
          const int q0 = qt_at(I, i) * BM;
          // The previous bulk reduction must have finished reading the staging tile.
          if (leader) {
            bulk_wait_read0();
            mbar_arrive(BAR(C::B_STGFREE));
          }
          if (!wait_warp(BAR(C::B_STGFREE), g & 1, ab, (kKBwdKV << 8) | 12)) {
            ok = false;
            break;
          }
          if constexpr (C::DQ_T) {
            // lanes = d index lr, columns = query q: 32 lanes write 128 contiguous bytes of row q
#pragma unroll
            for (int q = 0; q < COLS; ++q) stg[q * D + dq_swz(q, lr)] = __uint_as_float(v[q]);
          } else {
            // lanes = query row lr, columns = d
#pragma unroll
            for (int c = 0; c < COLS; c += 4)
              *reinterpret_cast<float4*>(stg + lr * D + dq_swz(lr, c)) =
                  make_float4(__uint_as_float(v[c]), __uint_as_float(v[c + 1]), __uint_as_float(v[c + 2]),
                              __uint_as_float(v[c + 3]));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C::B_STGFULL));
          bool lok = true;
          if (leader) {
            lok = wait_one(BAR(C::B_STGFULL), g & 1, ab, (kKBwdKV << 8) | 13);
            if (lok) {
              bulk_reduce_add_f32(p.dqacc + ((size_t)I.bh * p.Npad + q0) * D, smem_u32(stg), C::STG_BYTES);
              bulk_commit();
            }
          }
          if (!__all_sync(0xffffffffu, lok)) {  // the whole warp leaves together
            ok = false;
            break;
          }
        }
      }
      if (leader) bulk_wait0();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// --------------------------------------------------------------- dQ kernel
// 7-GEMM second kernel: CTA = 128 query rows of one head (M = query), walking
// its K/V tiles in the same direction as the forward:
//   S = Q K^T, dP = dO V^T (TMEM fp32), dS = P o (dP - D) (thread = query row)
//   written back as bf16 over dP's columns, then dQ += dS K (A = dS from TMEM,
//   B = K MN-major).  dQ * scale is written once at the end.
struct BwdQParams {
  CUtensorMap q_map;   // box {64, 128, 1}
  CUtensorMap do_map;  // box {64, 128, 1}
  CUtensorMap k_map;   // box {64, BN, 1}
  CUtensorMap v_map;   // box {64, BN, 1}
  const uint16_t* dO;  // bf16 [BH, N, hd] (read row by row into TMEM by DT configurations)
  const float* lse2;
  const float* dd;
  uint16_t* dq;
  int* err;
  int N, Npad, BH;
  int hd;  // head dim of the tensors (<= D)
  float scale_log2;
  float scale;
  int causal;
  int group;   // heads per launch-order group
  int items;   // work items (query tiles x key parts x dQ column parts x heads); the grid is persistent over them
  int* sched;  // [1]: next unclaimed work item (zero at launch)
  // Key-range split (few heads, long sequences): each query tile's key tiles are
  // cut into `ksplit` contiguous parts, each a work item of its own.  With
  // ksplit > 1 an item writes its fp32 dQ sum over its part (without the scale)
  // to dqpart [ksplit][BH][Npad][D] instead of dq, and bwd_qsum_kernel adds the
  // parts.
  int ksplit;
  float* dqpart;
};

// Sum of the key-range parts of dQ: dQ = scale * sum_s dqpart[s] (parts in fixed
// order, so the result is reproducible), bf16.
struct QSumParams {
  const float* dqpart;
  uint16_t* dq;
  int* err;
  int N, Npad, BH, hd, D, parts;
  float scale;
};

static __global__ void __launch_bounds__(256) bwd_qsum_kernel(const QSumParams p) {
  grid_dep_wait();
  if (*reinterpret_cast<volatile const int*>(p.err) != 0) return;
  const int tpr = p.hd / 8;
  const long long g = (long long)blockIdx.x * 256 + threadIdx.x;
  const long long row = g / tpr;  // bh * N + i
  if (row >= (long long)p.BH * p.N) return;
  const int c = (int)(g - row * tpr) * 8;
  const int bh = (int)(row / p.N), i = (int)(row % p.N);
  const size_t off = ((size_t)bh * p.Npad + i) * p.D + c;
  const size_t stride = (size_t)p.BH * p.Npad * p.D;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < p.parts; ++s) {
    const float4* q4 = reinterpret_cast<const float4*>(p.dqpart + s * stride + off);
    const float4 x0 = q4[0], x1 = q4[1];
    a[0] += x0.x; a[1] += x0.y; a[2] += x0.z; a[3] += x0.w;
    a[4] += x1.x; a[5] += x1.y; a[6] += x1.z; a[7] += x1.w;
  }
  const float sc = p.scale;
  *reinterpret_cast<uint4*>(p.dq + (size_t)row * p.hd + c) =
      make_uint4(pack_bf16(a[0] * sc, a[1] * sc), pack_bf16(a[2] * sc, a[3] * sc), pack_bf16(a[4] * sc, a[5] * sc),
                 pack_bf16(a[6] * sc, a[7] * sc));
}

// DT: dO lives in TMEM (written by the compute warps, thread = query row) and
// dP = dO V^T takes A from TMEM; the shared memory this saves holds more K/V
// slots, and the MMA order becomes S(j+1) (once the compute warps hold S(j) in
// registers), dQ(j), dP(j+1), so that S(j+1) runs during the softmax of j.
// DQS: the dQ columns are cut into DQS parts, each a work item of its own that
// recomputes S, dP and dS for its query tile (head dim 384, where the whole dQ
// accumulator does not fit TMEM next to S, dP and dO).
template <int D_, int BN_, int STAGES_, bool DT_ = false, int DQS_ = 1>
struct BwdQCfg {
  static constexpr int D = D_, BN = BN_, STAGES = STAGES_, DQS = DQS_;
  static constexpr int DQW = D / DQS;  // dQ columns per work item
  static constexpr bool DT = DT_;
  static constexpr int PANELS = D / 64;
  static constexpr uint32_t Q_PANEL = 128 * 128;
  static constexpr uint32_t Q_TILE = PANELS * Q_PANEL;
  static constexpr uint32_t KV_PANEL = BN * 128;
  static constexpr uint32_t KV_TILE = PANELS * KV_PANEL;
  static constexpr uint32_t OFF_Q = 0, OFF_DO = Q_TILE, OFF_KV = (DT ? 1 : 2) * Q_TILE;
  static constexpr uint32_t OFF_EPI = OFF_KV + STAGES * KV_TILE;
  // dQ epilogue staging (2 KB per compute warp) where shared memory allows.
  static constexpr uint32_t EPI_BYTES = OFF_EPI + 4 * 2048 + 512 + 1024 <= 232448 ? 4 * 2048 : 0;
  static constexpr uint32_t OFF_BAR = OFF_EPI + EPI_BYTES;
  static constexpr int IQ = 4;  // claimed work items passed from the producer to the other roles
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KVFULL = 2, B_KVEMPTY = 2 + STAGES, B_SDP = 2 + 2 * STAGES,
                       B_DS = B_SDP + 1, B_DQ = B_DS + 1, B_DONE = B_DQ + 1, B_ITEMFULL = B_DONE + 1,
                       B_ITEMEMPTY = B_ITEMFULL + IQ, B_SCONS = B_ITEMEMPTY + IQ, B_DOREADY = B_SCONS + 1,
                       NBAR = B_DOREADY + 1;
  static constexpr int ITEM_READERS = 1 + 4;  // the MMA warp and the four compute warps
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 32 + 1024;
  static constexpr int T_S = 0, T_DP = BN, T_DQ = 2 * BN;
  static constexpr int T_DO = 2 * BN + DQW;  // DT: dO as packed bf16 pairs, D / 2 columns
  static constexpr int TMEM_USED = 2 * BN + DQW + (DT ? D / 2 : 0);
  static constexpr uint32_t TMEM_COLS = TMEM_USED <= 256 ? 256 : 512;
  static constexpr int THREADS = 256;
  static_assert(TMEM_USED <= 512 && SMEM_BYTES <= 232448, "budgets");
  static_assert(!DT || BN <= 64, "DT holds a whole S and dP row of the tile in registers");
  static_assert(DQW % 64 == 0 && DQW <= 256, "dQ MMA width: whole panels, N <= 256");
};

// FEW: the key-split instantiation (p.ksplit >= 1); the plain one keeps one key
// part per query tile as a constant.
template <class C, bool FEW>
__global__ void __launch_bounds__(C::THREADS, 1) bwd_q_kernel(const __grid_constant__ BwdQParams p) {
  constexpr int D = C::D, BN = C::BN, S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw_addr);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 4);
  volatile int* item_ring = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 16);
  const int warp = warp_id();
  const int lane = lane_id();
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(BAR(C::B_QFULL), 1);
    mbar_init(BAR(C::B_QEMPTY), 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(BAR(C::B_KVFULL + s), 1);
      mbar_init(BAR(C::B_KVEMPTY + s), 1);
    }
    mbar_init(BAR(C::B_SDP), 1);
    mbar_init(BAR(C::B_DS), 4);
    mbar_init(BAR(C::B_DQ), 1);
    mbar_init(BAR(C::B_DONE), 1);
    for (int k = 0; k < C::IQ; ++k) {
      mbar_init(BAR(C::B_ITEMFULL + k), 1);
      mbar_init(BAR(C::B_ITEMEMPTY + k), C::ITEM_READERS);
    }
    mbar_init(BAR(C::B_SCONS), 4);
    mbar_init(BAR(C::B_DOREADY), 4);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const CtaAbort ab{abort_flag, p.err};
  grid_dep_wait();
  // A kernel that gave up earlier left the error word set: do nothing.
  const bool skip = *reinterpret_cast<volatile int*>(p.err) != 0;

  // Persistent work loop.  Work item w = (query tile of 128 rows, head) in
  // launch order: heads grouped for L2 reuse of their K and V, and under the
  // causal mask the query tiles that see the most key tiles first.  The
  // producer claims items from a global counter one item ahead and passes them
  // to the other roles through a shared-memory ring; barrier phases run on
  // across items.
  const int n_qt = (p.N + 127) / 128;
  const int ksplit = FEW ? p.ksplit : 1;
  struct Item {
    int q0, bh, n, h, j0, part;  // first query row, head, key tiles, dQ column part, first key tile, key part
  };
  auto coords = [&](int w) {
    Item I;
    int t;
    grouped_order(w, n_qt * ksplit * C::DQS, p.BH, p.group, t, I.bh);
    I.h = t % C::DQS;
    t /= C::DQS;
    int qt = t / ksplit;
    I.part = t - qt * ksplit;
    if (p.causal) qt = n_qt - 1 - qt;
    I.q0 = qt * 128;
    const int last = p.causal ? min(I.q0 + 127, p.N - 1) : p.N - 1;
    const int nk = last / BN + 1;
    if constexpr (FEW) {
      I.j0 = (int)((long long)I.part * nk / ksplit);
      I.n = (int)((long long)(I.part + 1) * nk / ksplit) - I.j0;
    } else {
      I.j0 = 0;
      I.n = nk;
    }
    return I;
  };
  auto item_warp = [&](int t) -> int {
    const int k = t % C::IQ;
    if (!wait_warp(BAR(C::B_ITEMFULL + k), (t / C::IQ) & 1, ab, (kKBwdQ << 8) | 8)) return -1;
    const int w = item_ring[k];
    __syncwarp();
    if (lane == 0) mbar_arrive(BAR(C::B_ITEMEMPTY + k));
    return w;
  };

  if (!skip) {
    if (warp == 0) {
      if (lane == 0) {
        tma_prefetch_desc(&p.q_map);
        tma_prefetch_desc(&p.do_map);
        tma_prefetch_desc(&p.k_map);
        tma_prefetch_desc(&p.v_map);
        int it = 0, nitems = 0, published = 0;
        bool ok = true;
        auto publish = [&](int w) -> bool {
          const int k = published % C::IQ;
          if (!wait_one(BAR(C::B_ITEMEMPTY + k), ((published / C::IQ) & 1) ^ 1, ab, (kKBwdQ << 8) | 9))
            return false;
          item_ring[k] = w;
          mbar_arrive(BAR(C::B_ITEMFULL + k));
          ++published;
          return true;
        };
        int wn = atomicAdd(p.sched + 1, 1);
        ok = publish(wn);
        while (ok && wn < p.items) {
          const Item I = coords(wn);
          wn = atomicAdd(p.sched + 1, 1);
          if (!publish(wn)) break;
          if (FEW && I.n == 0) continue;  // an empty key part: nothing to load or compute
          // The previous item's last S / dP MMAs must be done reading Q and dO.
          if (nitems > 0 && !wait_one(BAR(C::B_QEMPTY), (nitems - 1) & 1, ab, (kKBwdQ << 8) | 10)) break;
          mbar_expect_tx(BAR(C::B_QFULL), (C::DT ? 1 : 2) * C::Q_TILE);
          for (int pn = 0; pn < C::PANELS; ++pn) {
            tma_load_3d(sbase + C::OFF_Q + pn * C::Q_PANEL, &p.q_map, BAR(C::B_QFULL), 64 * pn, I.q0, I.bh);
            if (!C::DT)
              tma_load_3d(sbase + C::OFF_DO + pn * C::Q_PANEL, &p.do_map, BAR(C::B_QFULL), 64 * pn, I.q0, I.bh);
          }
          ++nitems;
          for (int j = 0; j < I.n && ok; ++j) {
            // The next item's Q and dO into L2 a few key steps before this item ends.
            if (j == max(0, I.n - 3) && wn < p.items) {
              const Item J = coords(wn);
              if (!FEW || J.n > 0)
                for (int pn = 0; pn < C::PANELS; ++pn) {
                  tma_prefetch_l2_3d(&p.q_map, 64 * pn, J.q0, J.bh);
                  tma_prefetch_l2_3d(&p.do_map, 64 * pn, J.q0, J.bh);
                }
            }
            for (int wkv = 0; wkv < 2; ++wkv) {
              const int s = it % S;
              if (!wait_one(BAR(C::B_KVEMPTY + s), ((it / S) & 1) ^ 1, ab, (kKBwdQ << 8) | 1)) {
                ok = false;
                break;
              }
              mbar_expect_tx(BAR(C::B_KVFULL + s), C::KV_TILE);
              const CUtensorMap* m = wkv ? &p.v_map : &p.k_map;
              for (int pn = 0; pn < C::PANELS; ++pn)
                tma_load_3d(sbase + C::OFF_KV + s * C::KV_TILE + pn * C::KV_PANEL, m, BAR(C::B_KVFULL + s),
                            64 * pn, (I.j0 + j) * BN, I.bh);
              if (j + 4 < I.n)
                for (int pn = 0; pn < C::PANELS; ++pn) tma_prefetch_l2_3d(m, 64 * pn, (I.j0 + j + 4) * BN, I.bh);
              ++it;
            }
          }
        }
        if (nitems > 0) wait_drain_bwd(BAR(C::B_QFULL), (nitems - 1) & 1);
        for (int i = max(0, it - S); i < it; ++i) wait_drain_bwd(BAR(C::B_KVFULL + i % S), (i / S) & 1);
      }
      __syncwarp();
    } else if (warp == 1) {
      // Whole warp; one elected lane issues (see mma_ss).
      constexpr uint32_t idS = make_idesc(128, BN, false, false);
      constexpr uint32_t idQ = make_idesc(128, C::DQW, false, true);
      bool ok = true;
      int it = 0, gj = 0, nitems = 0;
      if constexpr (C::DT) {
        auto kv_at = [&](int s) { return sbase + C::OFF_KV + s * C::KV_TILE; };
        // Next K or V slot in load order; false if the wait gave up.
        auto take = [&](int& slot) -> bool {
          slot = it % S;
          const bool got = wait_warp(BAR(C::B_KVFULL + slot), (it / S) & 1, ab, (kKBwdQ << 8) | 3);
          ++it;
          return got;
        };
        auto issue_s = [&](int sk) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss(tmem + C::T_S, desc_kmajor(sbase + C::OFF_Q, C::Q_PANEL, 16 * k),
                   desc_kmajor(kv_at(sk), C::KV_PANEL, 16 * k), idS, k > 0 ? 1u : 0u);
        };
        // dP = dO V^T with dO from TMEM (8 packed columns per 16 elements of d),
        // then the commits for the compute warps and for V's slot.
        auto issue_dp = [&](int sv) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ts(tmem + C::T_DP, tmem + C::T_DO + 8 * k, desc_kmajor(kv_at(sv), C::KV_PANEL, 16 * k), idS,
                   k > 0 ? 1u : 0u);
          mma_commit(BAR(C::B_SDP));
          mma_commit(BAR(C::B_KVEMPTY + sv));
        };
        for (int r = 0; ok; ++r) {
          const int w = item_warp(r);
          if (w < 0 || w >= p.items) break;
          const Item I = coords(w);
          if (FEW && I.n == 0) continue;
          if (!wait_warp(BAR(C::B_QFULL), nitems & 1, ab, (kKBwdQ << 8) | 2)) break;
          ++nitems;
          int sk = 0, sv = 0;
          // S(0) overwrites the previous item's last S, which the compute warps
          // have read once they arrive on SCONS for it.
          if (!take(sk) || !take(sv) ||
              (gj > 0 && !wait_warp(BAR(C::B_SCONS), (gj - 1) & 1, ab, (kKBwdQ << 8) | 11)))
            break;
          tc_fence_after();
          issue_s(sk);
          if (I.n == 1) mma_commit(BAR(C::B_QEMPTY));  // Q no longer read
          if (!wait_warp(BAR(C::B_DOREADY), (nitems - 1) & 1, ab, (kKBwdQ << 8) | 12)) break;
          tc_fence_after();
          issue_dp(sv);
          for (int j = 0; ok && j < I.n; ++j, ++gj) {
            const bool more = j + 1 < I.n;
            int sk1 = 0, sv1 = 0;
            if (more) {
              if (!take(sk1) || !take(sv1) || !wait_warp(BAR(C::B_SCONS), gj & 1, ab, (kKBwdQ << 8) | 11)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(sk1);
              if (j + 2 == I.n) mma_commit(BAR(C::B_QEMPTY));
            }
            if (!wait_warp(BAR(C::B_DS), gj & 1, ab, (kKBwdQ << 8) | 4)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t kq = kv_at(sk) + I.h * (C::DQW / 64) * C::KV_PANEL;  // this part's dQ columns of K
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)
              mma_ts(tmem + C::T_DQ, tmem + C::T_DP + 8 * k, desc_mnmajor(kq, C::KV_PANEL, 16 * k), idQ,
                     (j > 0 || k > 0) ? 1u : 0u);
            mma_commit(BAR(C::B_DQ));
            mma_commit(BAR(C::B_KVEMPTY + sk));
            // dP(j+1) overwrites dS(j) in dP's columns: issued after dQ(j), which reads it first.
            if (more) issue_dp(sv1);
            sk = sk1;
            sv = sv1;
          }
        }
      } else
      for (int r = 0; ok; ++r) {
        const int w = item_warp(r);
        if (w < 0 || w >= p.items) break;
        const Item I = coords(w);
        if (FEW && I.n == 0) continue;
        if (!wait_warp(BAR(C::B_QFULL), nitems & 1, ab, (kKBwdQ << 8) | 2)) break;
        ++nitems;
        for (int j = 0; ok && j < I.n; ++j, ++gj) {
          const int sk = it % S;
          if (!wait_warp(BAR(C::B_KVFULL + sk), (it / S) & 1, ab, (kKBwdQ << 8) | 3)) {
            ok = false;
            break;
          }
          ++it;
          const int sv = it % S;
          if (!wait_warp(BAR(C::B_KVFULL + sv), (it / S) & 1, ab, (kKBwdQ << 8) | 3)) {
            ok = false;
            break;
          }
          ++it;
          tc_fence_after();
          const uint32_t kb = sbase + C::OFF_KV + sk * C::KV_TILE;
          const uint32_t vb = sbase + C::OFF_KV + sv * C::KV_TILE;
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss(tmem + C::T_S, desc_kmajor(sbase + C::OFF_Q, C::Q_PANEL, 16 * k),
                   desc_kmajor(kb, C::KV_PANEL, 16 * k), idS, k > 0 ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss(tmem + C::T_DP, desc_kmajor(sbase + C::OFF_DO, C::Q_PANEL, 16 * k),
                   desc_kmajor(vb, C::KV_PANEL, 16 * k), idS, k > 0 ? 1u : 0u);
          mma_commit(BAR(C::B_SDP));
          mma_commit(BAR(C::B_KVEMPTY + sv));
          if (j + 1 == I.n) mma_commit(BAR(C::B_QEMPTY));  // Q and dO no longer read
          if (!wait_warp(BAR(C::B_DS), gj & 1, ab, (kKBwdQ << 8) | 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kq = kb + I.h * (C::DQW / 64) * C::KV_PANEL;  // this part's dQ columns of K
#pragma unroll
          for (int k = 0; k < BN / 16; ++k)
            mma_ts(tmem + C::T_DQ, tmem + C::T_DP + 8 * k, desc_mnmajor(kq, C::KV_PANEL, 16 * k), idQ,
                   (j > 0 || k > 0) ? 1u : 0u);
          mma_commit(BAR(C::B_DQ));
          mma_commit(BAR(C::B_KVEMPTY + sk));
        }
      }
      mma_commit(BAR(C::B_DONE));
      wait_drain_bwd(BAR(C::B_DONE), 0);
      __syncwarp();
    } else if (warp >= 4) {
      const int quad = warp & 3;
      const int r = quad * 32 + lane;
      const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
      const float cs = p.scale_log2;
      const float2 c2 = make_float2(cs, cs);
      bool ok = true;
      int gj = 0;
      for (int rr = 0; ok; ++rr) {
        const int w = item_warp(rr);
        if (w < 0 || w >= p.items) break;
        const Item I = coords(w);
        const int qi = I.q0 + r;
        // Key-split partial sums: [part][bh][Npad][D] fp32, this row's dQ columns.
        float* prow = nullptr;
        if constexpr (FEW)
          if (ksplit > 1)
            prow = p.dqpart + (((size_t)I.part * p.BH + I.bh) * p.Npad + qi) * D + I.h * C::DQW;
        if constexpr (FEW) {
          if (I.n == 0) {
            // An empty key part contributes zeros to the sum.
            if (prow != nullptr)
              for (int c = 0; c < C::DQW; c += 4) *reinterpret_cast<float4*>(prow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            continue;
          }
        }
        const float l2 = p.lse2[(size_t)I.bh * p.Npad + qi];  // -inf past N: every p is 0
        const float dd = p.dd[(size_t)I.bh * p.Npad + qi];
        const float2 l22 = make_float2(l2, l2), dd2 = make_float2(dd, dd);
        const int limit = p.causal ? min(qi, p.N - 1) : p.N - 1;
        if constexpr (C::DT) {
          // This item's dO row qi as packed bf16 pairs into TMEM lane r: the A
          // operand of dP = dO V^T.  The previous item's dP MMAs, the last readers
          // of these columns, completed before its last SDP barrier, which these
          // warps have waited on.
          const uint16_t* drow = p.dO + ((size_t)I.bh * p.N + (qi < p.N ? qi : 0)) * p.hd;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 64) {
            uint32_t ow[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              uint4 x = make_uint4(0u, 0u, 0u, 0u);
              if (qi < p.N && c0 + 8 * u < p.hd) x = *reinterpret_cast<const uint4*>(drow + c0 + 8 * u);
              ow[4 * u] = x.x;
              ow[4 * u + 1] = x.y;
              ow[4 * u + 2] = x.z;
              ow[4 * u + 3] = x.w;
            }
            tmem_st_32x32b_x32(trow + C::T_DO + (c0 >> 1), ow);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C::B_DOREADY));
        }
        for (int j = 0; j < I.n; ++j, ++gj) {
          if (!wait_warp(BAR(C::B_SDP), gj & 1, ab, (kKBwdQ << 8) | 5)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int kbase = (I.j0 + j) * BN;
          // P = exp2(S c - lse2) and dS = P (dP - D) for columns [c0, c0 + 32),
          // packed to bf16 over the first half of dP's columns (chunk c0 -> c0 / 2).
          auto ds_chunk = [&](int c0, const uint32_t* sr, const uint32_t* dr) {
            uint32_t pk[16];
            const bool masked = kbase + c0 + 31 > limit;
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 x = ffma2(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2, l22);
              float2 pe = make_float2(ex2(x.x), ex2(x.y));
              if (masked) {
                if (kbase + c0 + e > limit) pe.x = 0.f;
                if (kbase + c0 + e + 1 > limit) pe.y = 0.f;
              }
              const float2 ds =
                  fmul2(pe, fadd2(make_float2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), dd2));
              pk[e >> 1] = pack_bf16(ds.x, ds.y);
            }
            tmem_st_32x32b_x16(trow + C::T_DP + (c0 >> 1), pk);
          };
          if constexpr (C::DT) {
            // All of S into registers first: S(j+1) may then be issued over it.
            uint32_t sr[BN], dr[BN];
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32) tmem_ld_32x32b_x32(trow + C::T_S + c0, sr + c0);
            tmem_wait_ld();
            reg_fence<BN>(sr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::B_SCONS));
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32) tmem_ld_32x32b_x32(trow + C::T_DP + c0, dr + c0);
            tmem_wait_ld();
            reg_fence<BN>(dr);
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32) ds_chunk(c0, sr + c0, dr + c0);
          } else {
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32) {
              uint32_t sr[32], dr[32];
              tmem_ld_32x32b_x32(trow + C::T_S + c0, sr);
              tmem_ld_32x32b_x32(trow + C::T_DP + c0, dr);
              tmem_wait_ld();
              reg_fence<32>(sr);
              reg_fence<32>(dr);
              ds_chunk(c0, sr, dr);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C::B_DS));
        }
        if (!ok) break;
        // dQ epilogue; its TMEM reads finish before these warps arrive on DS for
        // the next item's first key tile, whose dQ MMA overwrites the accumulator.
        if (!wait_warp(BAR(C::B_DQ), (gj - 1) & 1, ab, (kKBwdQ << 8) | 6)) break;
        tc_fence_after();
        if constexpr (FEW) {
          if (prow != nullptr) {
            // Unscaled fp32 partial of this key part, every row of the tile (rows
            // past N are zero and never summed).
#pragma unroll
            for (int c0 = 0; c0 < C::DQW; c0 += 32) {
              uint32_t rv[32];
              tmem_ld_32x32b_x32(trow + C::T_DQ + c0, rv);
              tmem_wait_ld();
              reg_fence<32>(rv);
              float4* d4 = reinterpret_cast<float4*>(prow + c0);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                d4[v] = make_float4(__uint_as_float(rv[4 * v]), __uint_as_float(rv[4 * v + 1]),
                                    __uint_as_float(rv[4 * v + 2]), __uint_as_float(rv[4 * v + 3]));
            }
            tc_fence_before();
            continue;
          }
        }
        const int row0 = I.q0 + quad * 32;
        uint16_t* obase = p.dq + ((size_t)I.bh * p.N + (size_t)row0) * p.hd + I.h * C::DQW;
        const int hd_left = p.hd - I.h * C::DQW;  // columns of this part inside the head dim
        uint8_t* epi = gbase + C::OFF_EPI + quad * 2048;
#pragma unroll
        for (int c0 = 0; c0 < C::DQW; c0 += 32) {
          uint32_t rv[32];
          tmem_ld_32x32b_x32(trow + C::T_DQ + c0, rv);
          tmem_wait_ld();
          reg_fence<32>(rv);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            pk[e >> 1] = pack_bf16(__uint_as_float(rv[e]) * p.scale, __uint_as_float(rv[e + 1]) * p.scale);
          if constexpr (C::EPI_BYTES > 0) {
            // Staged: each warp store covers 8 rows x 64 contiguous bytes.
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<uint4*>(epi + lane * 64 + ((u ^ ((lane >> 1) & 3)) << 4)) =
                  make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            __syncwarp();
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int ri = jj * 8 + (lane >> 2), u = lane & 3;
              const uint4 val = *reinterpret_cast<const uint4*>(epi + ri * 64 + ((u ^ ((ri >> 1) & 3)) << 4));
              if (row0 + ri < p.N && c0 + 8 * u < hd_left)
                *reinterpret_cast<uint4*>(obase + (size_t)ri * p.hd + c0 + 8 * u) = val;
            }
            __syncwarp();
          } else {
            if (qi < p.N) {
              uint4* o4 = reinterpret_cast<uint4*>(obase + (size_t)lane * p.hd + c0);
#pragma unroll
              for (int v = 0; v < 4; ++v)
                if (c0 + 8 * v < hd_left) o4[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
          }
        }
        tc_fence_before();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace fa
