// Fused attention forward: O = softmax(scale * Q K^T) V and the per-row
// log-sum-exp, with no N x N matrix in HBM.
//
// Method ("ELI5: FlashAttention", tiling and softmax-statistics passages): the
// score matrix is cut into tiles; each query row keeps a running maximum m and
// exponential sum l, and partial results are merged with the normalising
// factor exp(m_old - m_new).  Here the running maximum is kept in the log2
// domain (scores are multiplied by scale*log2(e) so exp becomes ex2), and the
// accumulated O is only rescaled when the row maximum grew by more than 8
// (a factor 256): between rescales the probabilities are computed against the
// stale maximum, which is exact in arithmetic and keeps every p <= 256.
//
// CTA = NQ query tiles of 128 rows sharing one stream of K/V tiles (BN keys).
//   warp 0        TMA producer: Q tiles once, then K_j, V_j through a ring of
//                 STAGES shared-memory slots (mbarrier full/empty pairs)
//   warp 1        TMEM allocator and tcgen05.mma issuer (the whole warp runs
//                 the loop, one elected lane issues):
//                 S_t = Q_t K_j^T (both K-major, smem x smem -> TMEM) and
//                 O_t += P_t V_j (P from TMEM, V MN-major from smem)
//   warps 4..     one warpgroup per query tile; thread r owns row r of the tile
//                 (TMEM lane r), so row max / row sum need no shuffles; P is
//                 written back as bf16 into the columns of S (tcgen05.st)
// The MMA issue order S_0(0) S_1(0) PV_0(0) S_0(1) PV_1(0) S_1(1) ... lets the
// tensor core work on one tile while the other tile's softmax runs.
//
// QT (d = 192 and 256): Q lives in TMEM (written row by row by the softmax
// warps) and S = Q K^T takes A from TMEM, so 64-key tiles run at the full MMA
// rate and the shared memory holds more K/V slots; each tile's S is
// double-buffered in TMEM and the order S_t(0) S_t(1) PV_t(0) S_t(2) PV_t(1) ...
// lets the softmax warps run from one key tile to the next without waiting for
// S.  K/V tiles are loaded in that order (K one step ahead of V).
//
// QSD (d = 384): Q stays in shared memory (its 192 packed TMEM columns do not fit
// next to the 384-column O), with the same double-buffered S and issue order as
// QT; the producer loads each item's Q and the last S MMA of an item frees it.
// O += P V runs as two MMAs of 192 columns (an MMA's N is at most 256).
//
// Split-KV (splits > 1): every query block becomes `splits` work items, item s
// covering part s of the block's key tiles.  An item ends with O_s = O / l
// normalised by its own sum (fp32) and its log2-domain log-sum-exp L_s = m + log2 l
// (-inf where no key of the part is visible to the row); fwd_merge_kernel then
// combines the parts with the same max/sum algebra as the online softmax.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"

namespace fa {

struct FwdParams {
  CUtensorMap q_map;  // 3-D {d, N, B*H} bf16, box {64, 128, 1}, 128-byte swizzle
  CUtensorMap k_map;  // same tensor shape, box {64, BN, 1}
  CUtensorMap v_map;
  const uint16_t* q;  // bf16 [B*H, N, d] (read row by row into TMEM by QT configurations)
  uint16_t* o;  // bf16 [B*H, N, d]
  int dv;       // head dim d of the tensors (<= the kernel's D; columns d..D-1 of the tiles read as 0)
  float* lse;   // fp32 [B*H, N]
  int* err;
  int N;
  int BH;
  float scale_log2;  // scale * log2(e)
  int causal;
  int group;  // heads per launch-order group
  int items;  // work items (query blocks x heads x splits); the grid is persistent over them
  int splits;    // key-range parts per query block (1: O and LSE are written directly)
  float* opart;  // splits > 1: fp32 [splits, B*H, N, d], part s of row i = O_s(i) / l_s(i)
  float* lpart;  // splits > 1: fp32 [splits, B*H, N], log2-domain L_s(i) (-inf: no visible key)
};

// Merge of split-KV parts: for each row, L = log2 sum_s 2^(L_s) and
// O = sum_s 2^(L_s - L) O_s (bf16), LSE = L ln 2 (natural log, fp32).
struct FwdMergeParams {
  const float* opart;
  const float* lpart;
  uint16_t* o;
  float* lse;
  int* err;
  long long rows;  // B*H*N
  int dv;          // head dim (a multiple of 8)
  int splits;
};

template <int D_, int NQ_, int BN_, int STAGES_, bool QT_ = false, bool QSD_ = false>
struct FwdCfg {
  static constexpr int D = D_, NQ = NQ_, BN = BN_, STAGES = STAGES_;
  static constexpr bool QT = QT_;    // Q in TMEM, S double-buffered
  static constexpr bool QSD = QSD_;  // Q in shared memory, S double-buffered
  static constexpr bool SD = QT || QSD;
  static constexpr int SB = SD ? 2 : 1;  // S buffers per query tile
  static constexpr int NPV = (D + 255) / 256;  // O += P V as NPV MMAs of PVN columns
  static constexpr int PVN = D / NPV;
  static constexpr int BM = 128;
  static constexpr int PREFETCH = STAGES / 2 + 2;  // K/V tiles ahead for L2 prefetch
  static constexpr int QPF = 3;  // key steps before an item's end at which the next item's Q is prefetched
  static constexpr int PANELS = D / 64;
  static constexpr uint32_t Q_PANEL = BM * 128;
  static constexpr uint32_t Q_TILE = PANELS * Q_PANEL;
  static constexpr uint32_t KV_PANEL = BN * 128;
  static constexpr uint32_t KV_TILE = PANELS * KV_PANEL;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_KV = OFF_Q + (QT ? 0 : NQ * Q_TILE);
  // O epilogue staging: 2 KB per softmax warp (32 rows x 32 bf16 columns).
  static constexpr uint32_t OFF_EPI = OFF_KV + STAGES * KV_TILE;
  static constexpr uint32_t OFF_BAR = OFF_EPI + NQ * 4 * 2048;
  // barriers: q_full, kv_full[S], kv_empty[S], s_full[NQ*SB], p_ready[NQ*SB], o_ready[NQ*SB], done,
  // q_empty, q_ready (QT: Q written to TMEM).  With two S buffers, PV(j) commits to o_ready of
  // buffer j & 1: S(j+1) is issued ahead of PV(j), so one barrier for all PVs could trail a
  // waiter by two phases, which a parity wait cannot tell apart.
  static constexpr int B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = 1 + STAGES,
                       B_SFULL = 1 + 2 * STAGES, B_PREADY = B_SFULL + NQ * SB,
                       B_OREADY = B_PREADY + NQ * SB, B_DONE = B_OREADY + NQ * SB, B_QEMPTY = B_DONE + 1,
                       B_QREADY = B_QEMPTY + 1, NBAR = B_QREADY + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static constexpr int TMEM_S = 0;              // S_t (and P_t aliased) at (t*SB + buffer)*BN
  static constexpr int TMEM_O = NQ * SB * BN;   // O_t at TMEM_O + t*D
  static constexpr int TMEM_Q = TMEM_O + NQ * D;  // QT: Q_t as packed bf16 pairs at TMEM_Q + t*D/2
  static constexpr int TMEM_USED = TMEM_Q + (QT ? NQ * D / 2 : 0);
  static constexpr uint32_t TMEM_COLS =
      TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128 : TMEM_USED <= 256 ? 256 : 512;
  static constexpr int THREADS = 128 + 128 * NQ;
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static_assert(BN % 32 == 0 && BN <= 256 && D % 64 == 0 && D <= 384 && PVN % 64 == 0, "tile shape");
  static_assert(!(QT && QSD), "Q lives in one place");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

__device__ __forceinline__ int fwd_kv_tiles(int qrow0, int N, int causal, int BN) {
  if (qrow0 >= N) return 0;
  if (!causal) return (N + BN - 1) / BN;
  const int last = min(qrow0 + 127, N - 1);
  return last / BN + 1;
}

// Bounded wait used only while draining in-flight copies at teardown; it does
// not give up early when the CTA is aborting.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_test(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

// SPLIT: the split-KV instantiation (p.splits > 1); the plain one keeps lo = 0
// and s = 0 as constants and has no part epilogue.
template <class C, bool SPLIT>
__global__ void __launch_bounds__(C::THREADS, 1) fwd_kernel(const __grid_constant__ FwdParams p) {
  constexpr int D = C::D, NQ = C::NQ, BN = C::BN, S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw_addr);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_MISC + 4);
  const int warp = warp_id();
  const int lane = lane_id();

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar0 + 8 * C::B_QFULL, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bar0 + 8 * (C::B_KVFULL + s), 1);
      mbar_init(bar0 + 8 * (C::B_KVEMPTY + s), 1);
    }
    for (int t = 0; t < NQ * C::SB; ++t) {
      mbar_init(bar0 + 8 * (C::B_SFULL + t), 1);
      mbar_init(bar0 + 8 * (C::B_PREADY + t), 4);
      mbar_init(bar0 + 8 * (C::B_OREADY + t), 1);
    }
    mbar_init(bar0 + 8 * C::B_DONE, 1);
    mbar_init(bar0 + 8 * C::B_QEMPTY, 1);
    mbar_init(bar0 + 8 * C::B_QREADY, 4 * NQ);
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

  // Persistent work loop.  Work item w is (query block, head) in launch order:
  // heads grouped for L2 reuse, and under the causal mask the query blocks with
  // the most key tiles first.  CTA c takes items in "snake" order over rounds
  // (c, 2G-1-c, 2G+c, ...) so heavy and light items even out across CTAs.
  // Barrier phases run on across items: every role counts the same iterations.
  const int n_qblk = (p.N + 128 * NQ - 1) / (128 * NQ);
  auto item_of = [&](int r) -> int {
    const int G = gridDim.x, c = blockIdx.x;
    return r * G + ((r & 1) ? (G - 1 - c) : c);
  };
  // Item w: query block and head from w / splits, key part s = w % splits.
  // Part s of a block whose tiles see nf key tiles at most is tiles
  // [s*nf/splits, (s+1)*nf/splits); nkv[t] counts those tile t sees (may be 0).
  struct Item {
    int q0, bh, nmax;
    int nkv[NQ];
  };
  struct Part {
    int s, lo;
  };
  auto coords = [&](int w) {
    Item it;
    int qb;
    const int wb = SPLIT ? w / p.splits : w;
    grouped_order(wb, n_qblk, p.BH, p.group, qb, it.bh);
    if (p.causal) qb = n_qblk - 1 - qb;
    it.q0 = qb * 128 * NQ;
    it.nmax = 0;
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
      it.nkv[t] = fwd_kv_tiles(it.q0 + 128 * t, p.N, p.causal, BN);
      it.nmax = max(it.nmax, it.nkv[t]);
    }
    if constexpr (SPLIT) {
      const int s = w - wb * p.splits;
      const int nf = it.nmax;
      const int lo = (int)((long long)s * nf / p.splits);
      const int hi = (int)((long long)(s + 1) * nf / p.splits);
      it.nmax = 0;
#pragma unroll
      for (int t = 0; t < NQ; ++t) {
        it.nkv[t] = max(0, min(hi, it.nkv[t]) - lo);
        it.nmax = max(it.nmax, it.nkv[t]);
      }
    }
    return it;
  };
  // Split instantiation: part index s of item w and its first key tile.
  auto part_of = [&](int w) {
    Part pt{0, 0};
    if constexpr (SPLIT) {
      const int wb = w / p.splits;
      pt.s = w - wb * p.splits;
      int qb, bh;
      grouped_order(wb, n_qblk, p.BH, p.group, qb, bh);
      if (p.causal) qb = n_qblk - 1 - qb;
      int nf = 0;
#pragma unroll
      for (int t = 0; t < NQ; ++t) nf = max(nf, fwd_kv_tiles(qb * 128 * NQ + 128 * t, p.N, p.causal, BN));
      pt.lo = (int)((long long)pt.s * nf / p.splits);
    }
    return pt;
  };
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };

  // Two softmax warpgroups (384 threads, 168 registers each at launch): the
  // producer/MMA warpgroup gives registers to the softmax warpgroups;
  // 128 * 88 + 256 * 208 equals the 384 * 168 the block was launched with.
  constexpr bool kSplitRegs = C::THREADS == 384;
  if (!skip) {
    if (warp < 4) {
    if constexpr (kSplitRegs) regs_shrink<88>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        tma_prefetch_desc(&p.q_map);
        tma_prefetch_desc(&p.k_map);
        tma_prefetch_desc(&p.v_map);
        int it = 0, nitems = 0;
        bool ok = true;
        // No L2 prefetches until the CTA's first K tile has landed (at the start
        // every CTA loads at once; prefetches then only delay the first tiles).
        // Slot 0 has seen one load until more than S were issued, and the (S+1)-th
        // waited for the first to be consumed.
        bool warm = false;
        auto is_warm = [&]() -> bool {
          if (!warm) warm = it > S || (it >= 1 && mbar_test(BAR(C::B_KVFULL), 0));
          return warm;
        };
        for (int r = 0; ok; ++r) {
          const int w = item_of(r);
          if (w >= p.items) break;
          const Item I = coords(w);
          const Part P = part_of(w);
          // The next item's Q tiles into L2 a few key steps before this item ends,
          // so that its load (or, with Q in TMEM, the softmax warps' row reads)
          // at the item change is served from L2.
          auto prefetch_next_q = [&](int j) {
            if (j != max(0, I.nmax - C::QPF) || !is_warm()) return;
            const int w2 = item_of(r + 1);
            if (w2 >= p.items) return;
            const Item J = coords(w2);
            for (int t = 0; t < NQ; ++t)
              if (J.q0 + 128 * t < p.N)
                for (int pn = 0; pn < C::PANELS; ++pn) tma_prefetch_l2_3d(&p.q_map, 64 * pn, J.q0 + 128 * t, J.bh);
          };
          if constexpr (C::SD) {
            if (C::QSD && I.nmax > 0) {
              // This item's Q, once the previous item's S MMAs are done reading Q.
              if (!wait_one(BAR(C::B_QEMPTY), (nitems & 1) ^ 1, ab, (kKFwd << 8) | 10)) break;
              mbar_expect_tx(BAR(C::B_QFULL), NQ * C::Q_TILE);
              for (int t = 0; t < NQ; ++t)
                for (int pn = 0; pn < C::PANELS; ++pn)
                  tma_load_3d(sbase + C::OFF_Q + t * C::Q_TILE + pn * C::Q_PANEL, &p.q_map, BAR(C::B_QFULL), 64 * pn,
                              I.q0 + 128 * t, I.bh);
              ++nitems;
            }
            // K(0), then K(j+1) ahead of V(j): the order in which the MMAs read them.
            auto load = [&](const CUtensorMap* m, int j) -> bool {
              const int s = it % S;
              if (!wait_one(BAR(C::B_KVEMPTY + s), ((it / S) & 1) ^ 1, ab, (kKFwd << 8) | 1)) return false;
              mbar_expect_tx(BAR(C::B_KVFULL + s), C::KV_TILE);
              for (int pn = 0; pn < C::PANELS; ++pn)
                tma_load_3d(sbase + C::OFF_KV + s * C::KV_TILE + pn * C::KV_PANEL, m, BAR(C::B_KVFULL + s),
                            64 * pn, (P.lo + j) * BN, I.bh);
              if (j + C::PREFETCH < I.nmax && is_warm())
                for (int pn = 0; pn < C::PANELS; ++pn)
                  tma_prefetch_l2_3d(m, 64 * pn, (P.lo + j + C::PREFETCH) * BN, I.bh);
              ++it;
              return true;
            };
            if (I.nmax > 0) ok = load(&p.k_map, 0);
            for (int j = 0; j < I.nmax && ok; ++j) {
              prefetch_next_q(j);
              if (j + 1 < I.nmax) ok = load(&p.k_map, j + 1);
              if (ok) ok = load(&p.v_map, j);
            }
            continue;
          }
          if (SPLIT && I.nmax == 0) continue;  // an empty key part: nothing to load or compute
          // The previous item's S MMAs must be done reading Q.
          if (!wait_one(BAR(C::B_QEMPTY), (nitems & 1) ^ 1, ab, (kKFwd << 8) | 10)) break;
          mbar_expect_tx(BAR(C::B_QFULL), NQ * C::Q_TILE);
          for (int t = 0; t < NQ; ++t)
            for (int pn = 0; pn < C::PANELS; ++pn)
              tma_load_3d(sbase + C::OFF_Q + t * C::Q_TILE + pn * C::Q_PANEL, &p.q_map, BAR(C::B_QFULL), 64 * pn,
                          I.q0 + 128 * t, I.bh);
          ++nitems;
          for (int j = 0; j < I.nmax && ok; ++j) {
            prefetch_next_q(j);
            for (int wkv = 0; wkv < 2; ++wkv) {
              const int s = it % S;
              if (!wait_one(BAR(C::B_KVEMPTY + s), ((it / S) & 1) ^ 1, ab, (kKFwd << 8) | 1)) {
                ok = false;
                break;
              }
              mbar_expect_tx(BAR(C::B_KVFULL + s), C::KV_TILE);
              const CUtensorMap* m = wkv ? &p.v_map : &p.k_map;
              for (int pn = 0; pn < C::PANELS; ++pn)
                tma_load_3d(sbase + C::OFF_KV + s * C::KV_TILE + pn * C::KV_PANEL, m, BAR(C::B_KVFULL + s),
                            64 * pn, (P.lo + j) * BN, I.bh);
              // Pull K/V tiles a few steps beyond the ring into L2.
              if (j + C::PREFETCH < I.nmax && is_warm())
                for (int pn = 0; pn < C::PANELS; ++pn)
                  tma_prefetch_l2_3d(m, 64 * pn, (P.lo + j + C::PREFETCH) * BN, I.bh);
              ++it;
            }
          }
        }
        // Let every copy this thread started land before the CTA can exit.
        if (nitems > 0) wait_drain(BAR(C::B_QFULL), (nitems - 1) & 1);
        for (int i = max(0, it - S); i < it; ++i) wait_drain(BAR(C::B_KVFULL + i % S), (i / S) & 1);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issue
      {
        constexpr uint32_t idS = make_idesc(128, BN, false, false);
        constexpr uint32_t idO = make_idesc(128, C::PVN, false, true);
        // O_t (+)= P V over the 16-key step k, as NPV MMAs of PVN columns each.
        auto issue_pv = [&](int t, uint32_t p_tmem, uint32_t vb, int k, uint32_t acc) {
#pragma unroll
          for (int c = 0; c < C::NPV; ++c)
            mma_ts(tmem + C::TMEM_O + t * D + c * C::PVN, p_tmem,
                   desc_mnmajor(vb + c * (C::PVN / 64) * C::KV_PANEL, C::KV_PANEL, 16 * k), idO, acc);
        };
        auto issue_s = [&](int t, int s) {
          const uint32_t qa = sbase + C::OFF_Q + t * C::Q_TILE;
          const uint32_t kb = sbase + C::OFF_KV + s * C::KV_TILE;
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss(tmem + C::TMEM_S + t * BN, desc_kmajor(qa, C::Q_PANEL, 16 * k),
                   desc_kmajor(kb, C::KV_PANEL, 16 * k), idS, k > 0 ? 1u : 0u);
          mma_commit(BAR(C::B_SFULL + t));
        };
        int it = 0, nitems = 0;
        int g[NQ];
#pragma unroll
        for (int t = 0; t < NQ; ++t) g[t] = 0;
        bool ok = true;
        if constexpr (C::SD) {
          // Next K or V slot in load order (false if the wait gave up).
          auto take = [&](int& slot) -> bool {
            slot = it % S;
            const bool got = wait_warp(BAR(C::B_KVFULL + slot), (it / S) & 1, ab, (kKFwd << 8) | 3);
            ++it;
            return got;
          };
          // S_t into buffer b of tile t with A = Q_t from TMEM (8 packed columns per
          // 16 elements of d).
          auto issue_sq = [&](int t, int b, int sk) {
            const uint32_t kb = sbase + C::OFF_KV + sk * C::KV_TILE;
            if constexpr (C::QT) {
#pragma unroll
              for (int k = 0; k < D / 16; ++k)
                mma_ts(tmem + C::TMEM_S + (t * C::SB + b) * BN, tmem + C::TMEM_Q + t * (D / 2) + 8 * k,
                       desc_kmajor(kb, C::KV_PANEL, 16 * k), idS, k > 0 ? 1u : 0u);
            } else {
              const uint32_t qa = sbase + C::OFF_Q + t * C::Q_TILE;
#pragma unroll
              for (int k = 0; k < D / 16; ++k)
                mma_ss(tmem + C::TMEM_S + (t * C::SB + b) * BN, desc_kmajor(qa, C::Q_PANEL, 16 * k),
                       desc_kmajor(kb, C::KV_PANEL, 16 * k), idS, k > 0 ? 1u : 0u);
            }
            mma_commit(BAR(C::B_SFULL + t * C::SB + b));
          };
          for (int r = 0; ok; ++r) {
            const int w = item_of(r);
            if (w >= p.items) break;
            const Item I = coords(w);
            // An empty key part has no Q hand-off (the softmax warps skip it too).
            if (I.nmax <= 0) continue;
            // QT: the softmax warps have written this item's Q into TMEM; QSD: its TMA load landed.
            if (!wait_warp(BAR(C::QT ? C::B_QREADY : C::B_QFULL), nitems & 1, ab, (kKFwd << 8) | 11)) break;
            ++nitems;
            int sk = 0;
            if (!take(sk)) break;
            tc_fence_after();
            for (int t = 0; t < NQ; ++t)
              if (I.nkv[t] > 0) issue_sq(t, g[t] & 1, sk);
            mma_commit(BAR(C::B_KVEMPTY + sk));
            if (C::QSD && I.nmax == 1) mma_commit(BAR(C::B_QEMPTY));  // the item's last S MMAs
            for (int j = 0; ok && j < I.nmax; ++j) {
              // S_t(j+1) into the other buffer of tile t, whose P_t(j-1) was read by
              // PV_t(j-1) (issued before).
              if (j + 1 < I.nmax) {
                if (!take(sk)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                for (int t = 0; t < NQ; ++t)
                  if (j + 1 < I.nkv[t]) issue_sq(t, (g[t] + j + 1) & 1, sk);
                mma_commit(BAR(C::B_KVEMPTY + sk));
                if (C::QSD && j + 2 == I.nmax) mma_commit(BAR(C::B_QEMPTY));  // the item's last S MMAs
              }
              int sv = 0;
              if (!take(sv)) {
                ok = false;
                break;
              }
              const uint32_t vb = sbase + C::OFF_KV + sv * C::KV_TILE;
              for (int t = 0; t < NQ && ok; ++t) {
                if (j >= I.nkv[t]) continue;
                const int gj = g[t] + j;
                const int sb = t * C::SB + (gj & 1);
                if (!wait_warp(BAR(C::B_PREADY + sb), (gj >> 1) & 1, ab, (kKFwd << 8) | 5)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                  issue_pv(t, tmem + C::TMEM_S + sb * BN + 8 * k, vb, k, (j > 0 || k > 0) ? 1u : 0u);
                mma_commit(BAR(C::B_OREADY + sb));
              }
              if (!ok) break;
              mma_commit(BAR(C::B_KVEMPTY + sv));
            }
#pragma unroll
            for (int t = 0; t < NQ; ++t) g[t] += I.nkv[t];
          }
        } else
        for (int r = 0; ok; ++r) {
          const int w = item_of(r);
          if (w >= p.items) break;
          const Item I = coords(w);
          if (SPLIT && I.nmax == 0) continue;  // an empty key part (the producer loaded nothing)
          ok = wait_warp(BAR(C::B_QFULL), nitems & 1, ab, (kKFwd << 8) | 2);
          ++nitems;
          if (!ok) break;
          {
            const int s = it % S;
            ok = wait_warp(BAR(C::B_KVFULL + s), (it / S) & 1, ab, (kKFwd << 8) | 3);
            if (!ok) break;
            tc_fence_after();
            for (int t = 0; t < NQ; ++t)
              if (I.nkv[t] > 0) issue_s(t, s);
            mma_commit(BAR(C::B_KVEMPTY + s));
            if (I.nmax == 1) mma_commit(BAR(C::B_QEMPTY));
            ++it;
          }
          for (int j = 0; ok && j < I.nmax; ++j) {
            const int sv = it % S;
            ok = wait_warp(BAR(C::B_KVFULL + sv), (it / S) & 1, ab, (kKFwd << 8) | 4);
            ++it;
            if (!ok) break;
            tc_fence_after();
            const int sk = it % S;
            bool k_ready = false;
            const uint32_t vb = sbase + C::OFF_KV + sv * C::KV_TILE;
            for (int t = 0; t < NQ && ok; ++t) {
              if (j < I.nkv[t]) {
                if (!wait_warp(BAR(C::B_PREADY + t), (g[t] + j) & 1, ab, (kKFwd << 8) | 5)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                  issue_pv(t, tmem + C::TMEM_S + t * BN + 8 * k, vb, k, (j > 0 || k > 0) ? 1u : 0u);
                mma_commit(BAR(C::B_OREADY + t));
              }
              if (j + 1 < I.nkv[t]) {
                if (!k_ready) {
                  if (!wait_warp(BAR(C::B_KVFULL + sk), (it / S) & 1, ab, (kKFwd << 8) | 6)) {
                    ok = false;
                    break;
                  }
                  tc_fence_after();
                  k_ready = true;
                }
                issue_s(t, sk);
              }
            }
            if (!ok) break;
            mma_commit(BAR(C::B_KVEMPTY + sv));
            if (k_ready) {
              mma_commit(BAR(C::B_KVEMPTY + sk));
              ++it;
            }
            // The item's last S MMAs have been issued: Q may be reloaded once they finish.
            if (j + 2 == I.nmax) mma_commit(BAR(C::B_QEMPTY));
          }
#pragma unroll
          for (int t = 0; t < NQ; ++t) g[t] += I.nkv[t];
        }
        // Every MMA issued above must finish before TMEM is released.
        mma_commit(BAR(C::B_DONE));
        wait_drain(BAR(C::B_DONE), 0);
      }
      __syncwarp();
    }
    } else {
      // ------------------------------------------------------------ softmax
      if constexpr (kSplitRegs) regs_grow<208>();
      const int t = (warp - 4) >> 2;
      const int quad = warp & 3;
      const int r = quad * 32 + lane;
      const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
      const uint32_t tO = trow + C::TMEM_O + t * D;
      const float cs = p.scale_log2;
      // Barrier and phase parity that signal completion of this tile's gm-th PV.
      auto oready_bar = [&](int gm) { return C::SD ? t * C::SB + (gm & 1) : t; };
      auto oready_phase = [&](int gm) -> uint32_t { return C::SD ? ((gm >> 1) & 1) : (gm & 1); };
      int g = 0;  // iterations of this query tile in earlier items
      bool ok = true;
      // QT: item wq's query row r as packed bf16 pairs into TMEM lane r (the A
      // operand of S = Q K^T).  Called once the S MMAs of the previous item,
      // the last readers of these columns, are known to be complete.
      auto write_q = [&](int wq) {
        const Item J = coords(wq);
        const int qrow = J.q0 + 128 * t + r;
        const uint16_t* qsrc = p.q + ((size_t)J.bh * p.N + (qrow < p.N ? qrow : 0)) * p.dv;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 64) {
          uint32_t qw[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (qrow < p.N && c0 + 8 * u < p.dv) x = *reinterpret_cast<const uint4*>(qsrc + c0 + 8 * u);
            qw[4 * u] = x.x;
            qw[4 * u + 1] = x.y;
            qw[4 * u + 2] = x.z;
            qw[4 * u + 3] = x.w;
          }
          tmem_st_32x32b_x32(trow + C::TMEM_Q + t * (D / 2) + (c0 >> 1), qw);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::B_QREADY));
      };
      // QT: the first item at or after round r with key tiles (-1 if none).  Q is
      // written only for those: one QREADY phase per item the issuer waits for, so
      // the barrier never runs two phases ahead of its waiter.
      auto next_work = [&](int r0) -> int {
        if constexpr (!SPLIT) return item_of(r0) < p.items ? item_of(r0) : -1;
        for (int r2 = r0;; ++r2) {
          const int w2 = item_of(r2);
          if (w2 >= p.items) return -1;
          if (coords(w2).nmax > 0) return w2;
        }
      };
      for (int rr = 0; ok; ++rr) {
        const int w = item_of(rr);
        if (w >= p.items) break;
        if (C::QT && rr == 0) {
          const int wq = next_work(0);
          if (wq >= 0) write_q(wq);
        }
        const Item I = coords(w);
        const Part P = part_of(w);
        const int qi = I.q0 + 128 * t + r;
        const int n = I.nkv[t];
        const int bh = I.bh;
        const int limit = p.causal ? min(qi, p.N - 1) : p.N - 1;
        float m_used = -INFINITY;
        float l = 0.f;
        for (int j = 0; j < n; ++j) {
          // S buffer (and its barriers) of this step: per tile, or alternating (QT, QSD).
          const int sb = C::SD ? t * C::SB + ((g + j) & 1) : t;
          const uint32_t sph = C::SD ? (((g + j) >> 1) & 1) : ((g + j) & 1);
          const uint32_t tS = trow + C::TMEM_S + sb * BN;
          if (!wait_warp(BAR(C::B_SFULL + sb), sph, ab, (kKFwd << 8) | 7)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t sr[BN];
#pragma unroll
          for (int c = 0; c < BN; c += 32) tmem_ld_32x32b_x32(tS + c, sr + c);
          tmem_wait_ld();
          reg_fence<BN>(sr);
          const int kbase = (P.lo + j) * BN;
          if (kbase + BN - 1 > limit) {
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (kbase + c > limit) sr[c] = __float_as_uint(-INFINITY);
          }
          // Row maximum: four independent chains of three-input max.
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
          for (int c = 0; c < BN; c += 8) {
            mx0 = max3(mx0, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            mx1 = max3(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
            mx2 = max3(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
            mx3 = max3(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
          }
          const float m_cand = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * cs;
          const bool need = m_cand > m_used + 8.0f;
          float alpha = 1.f;
          if (need) {
            alpha = ex2(m_used - m_cand);
            m_used = m_cand;
            l *= alpha;
          }
          const float msub = (m_used == -INFINITY) ? 0.f : m_used;
          // p = exp2(s * c - m), two columns per packed FMA / add.
          const float2 c2 = make_float2(cs, cs), nm2 = make_float2(-msub, -msub);
          float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < BN; c += 32) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float2 x01 =
                  ffma2(make_float2(__uint_as_float(sr[c + e]), __uint_as_float(sr[c + e + 1])), c2, nm2);
              const float2 x23 =
                  ffma2(make_float2(__uint_as_float(sr[c + e + 2]), __uint_as_float(sr[c + e + 3])), c2, nm2);
              const float2 p01 = make_float2(ex2(x01.x), ex2(x01.y));
              const float2 p23 = make_float2(ex2(x23.x), ex2(x23.y));
              la = fadd2(la, p01);
              lb = fadd2(lb, p23);
              pk[e >> 1] = pack_bf16(p01.x, p01.y);
              pk[(e >> 1) + 1] = pack_bf16(p23.x, p23.y);
            }
            tmem_st_32x32b_x16(tS + (c >> 1), pk);
          }
          l += (la.x + la.y) + (lb.x + lb.y);
          tmem_wait_st();
          if (j > 0 && __any_sync(0xffffffffu, need)) {
            // Rescale the running O once the MMA that last accumulated into it is done.
            if (!wait_warp(BAR(C::B_OREADY + oready_bar(g + j - 1)), oready_phase(g + j - 1), ab, (kKFwd << 8) | 8)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t orr[32];
              tmem_ld_32x32b_x32(tO + c0, orr);
              tmem_wait_ld();
              reg_fence<32>(orr);
#pragma unroll
              for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
              tmem_st_32x32b_x32(tO + c0, orr);
            }
            tmem_wait_st();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(C::B_PREADY + sb));
        }
        if (C::QT && ok && I.nmax > 0) {
          const int wn = next_work(rr + 1);
          if (wn >= 0) write_q(wn);
        }
        if (ok && n > 0) {
          if (!wait_warp(BAR(C::B_OREADY + oready_bar(g + n - 1)), oready_phase(g + n - 1), ab, (kKFwd << 8) | 9)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool store = qi < p.N;
          // Staged through this warp's 2 KB of shared memory, 32 columns at a
          // time: each thread writes its row, then each warp store covers 8 rows
          // x 64 contiguous bytes instead of 32 rows x 16 bytes.
          uint8_t* epi = gbase + C::OFF_EPI + (t * 4 + quad) * 2048;
          const int row0 = I.q0 + 128 * t + quad * 32;  // this warp's first query row
          if constexpr (!SPLIT) {
            const float inv = 1.f / l;
            uint16_t* obase = p.o + ((size_t)bh * p.N + (size_t)row0) * p.dv;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t orr[32];
              tmem_ld_32x32b_x32(tO + c0, orr);
              tmem_wait_ld();
              reg_fence<32>(orr);
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 32; e += 2)
                pk[e >> 1] = pack_bf16(__uint_as_float(orr[e]) * inv, __uint_as_float(orr[e + 1]) * inv);
#pragma unroll
              for (int u = 0; u < 4; ++u)
                *reinterpret_cast<uint4*>(epi + lane * 64 + ((u ^ ((lane >> 1) & 3)) << 4)) =
                    make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int rr = j * 8 + (lane >> 2), u = lane & 3;
                const uint4 val = *reinterpret_cast<const uint4*>(epi + rr * 64 + ((u ^ ((rr >> 1) & 3)) << 4));
                if (row0 + rr < p.N && c0 + 8 * u < p.dv)
                  *reinterpret_cast<uint4*>(obase + (size_t)rr * p.dv + c0 + 8 * u) = val;
              }
              __syncwarp();
            }
            if (store) p.lse[(size_t)bh * p.N + qi] = (m_used + log2f(l)) * kLn2;
          } else {
            // Part s of a split-KV pass: fp32 O / l and the log2-domain L_s, staged
            // 16 columns (64 bytes per row) at a time.  A row that sees no key of
            // the part (l = 0) gets O_s = 0 and L_s = -inf.
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float* pbase = p.opart + (((size_t)P.s * p.BH + bh) * p.N + (size_t)row0) * p.dv;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t orr[32];
              tmem_ld_32x32b_x32(tO + c0, orr);
              tmem_wait_ld();
              reg_fence<32>(orr);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int e = 16 * h + 4 * u;
                  *reinterpret_cast<float4*>(epi + lane * 64 + ((u ^ ((lane >> 1) & 3)) << 4)) =
                      make_float4(__uint_as_float(orr[e]) * inv, __uint_as_float(orr[e + 1]) * inv,
                                  __uint_as_float(orr[e + 2]) * inv, __uint_as_float(orr[e + 3]) * inv);
                }
                __syncwarp();
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                  const int rr = jj * 8 + (lane >> 2), u = lane & 3;
                  const float4 val =
                      *reinterpret_cast<const float4*>(epi + rr * 64 + ((u ^ ((rr >> 1) & 3)) << 4));
                  const int col = c0 + 16 * h + 4 * u;
                  if (row0 + rr < p.N && col < p.dv)
                    *reinterpret_cast<float4*>(pbase + (size_t)rr * p.dv + col) = val;
                }
                __syncwarp();
              }
            }
            if (store)
              p.lpart[((size_t)P.s * p.BH + bh) * p.N + qi] = l > 0.f ? m_used + log2f(l) : -INFINITY;
          }
        } else if (SPLIT && ok && qi < p.N) {
          // This query tile sees no key tile of the part.
          p.lpart[((size_t)P.s * p.BH + bh) * p.N + qi] = -INFINITY;
        }
        g += n;
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

// Merge of the split-KV parts: one thread per 8 columns of a row.  Each thread
// reads the row's `splits` values of L_s (cached), so no shuffles are needed.
// A part with L_s = -inf saw no key of the row and is skipped (its O_s is
// not read).  Skipped entirely if a kernel gave up a wait.
__global__ void __launch_bounds__(256) fwd_merge_kernel(const __grid_constant__ FwdMergeParams p) {
  grid_dep_wait();
  if (*reinterpret_cast<volatile const int*>(p.err) != 0) return;
  const int tpr = p.dv / 8;
  const long long g = (long long)blockIdx.x * 256 + threadIdx.x;
  const long long row = g / tpr;
  if (row >= p.rows) return;
  const int c = (int)(g - row * tpr) * 8;
  float mx = -INFINITY;
  for (int s = 0; s < p.splits; ++s) mx = fmaxf(mx, p.lpart[(size_t)s * p.rows + row]);
  float wsum = 0.f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (mx != -INFINITY) {
    for (int s = 0; s < p.splits; ++s) {
      const float ls = p.lpart[(size_t)s * p.rows + row];
      if (ls == -INFINITY) continue;
      const float wt = exp2f(ls - mx);
      wsum += wt;
      const float* src = p.opart + ((size_t)s * p.rows + row) * p.dv + c;
      const float4 a = *reinterpret_cast<const float4*>(src);
      const float4 b = *reinterpret_cast<const float4*>(src + 4);
      acc[0] += wt * a.x;
      acc[1] += wt * a.y;
      acc[2] += wt * a.z;
      acc[3] += wt * a.w;
      acc[4] += wt * b.x;
      acc[5] += wt * b.y;
      acc[6] += wt * b.z;
      acc[7] += wt * b.w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint4 out;
  out.x = pack_bf16(acc[0] * inv, acc[1] * inv);
  out.y = pack_bf16(acc[2] * inv, acc[3] * inv);
  out.z = pack_bf16(acc[4] * inv, acc[5] * inv);
  out.w = pack_bf16(acc[6] * inv, acc[7] * inv);
  *reinterpret_cast<uint4*>(p.o + (size_t)row * p.dv + c) = out;
  if (c == 0) p.lse[row] = wsum > 0.f ? (mx + log2f(wsum)) * kLn2 : -INFINITY;
}

}  // namespace fa
