// Shared kernel infrastructure: bounded mbarrier waits that report a device
// error instead of hanging, and small numeric helpers.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fa {

// Device error word layout (two ints owned by the library per device):
//   err[0] = status (0 = ok, 6 = a bounded wait expired)
//   err[1] = where: (kernel id << 8) | wait site
constexpr int kDevErrTimeout = 6;
enum KernelId : int { kKFwd = 1, kKBwdKV = 2, kKBwdQ = 3, kKPre = 4, kKConv = 5, kKSelfTest = 6 };

// About two seconds at the maximum SM clock: far longer than any legitimate
// wait inside these kernels (microseconds), short enough to keep a broken
// launch from holding the GPU.
constexpr long long kWaitLimitCycles = 4000000000LL;

struct CtaAbort {
  volatile int* flag;  // shared memory; set once any wait in the CTA gave up
  int* gerr;           // global error word
};

__device__ __forceinline__ void raise_timeout(const CtaAbort& ab, int where) {
  *ab.flag = 1;
  if (atomicCAS(ab.gerr, 0, kDevErrTimeout) == 0) atomicExch(ab.gerr + 1, where);
}

// Single-thread bounded wait for the phase of `bar` with the given parity.
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, const CtaAbort& ab,
                                         int where) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_test(bar, parity)) return true;
    if (*ab.flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      raise_timeout(ab, where);
      return false;
    }
  }
}

// Warp-uniform bounded wait: every lane polls, and the warp proceeds only if all
// lanes saw the phase complete, so the warp-collective tcgen05 instructions that
// follow are executed by all lanes or by none.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const CtaAbort& ab,
                                          int where) {
  bool ok = wait_one(bar, parity, ab, where);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait until a shared-memory counter written by another warp of the
// CTA reaches `target`.
__device__ __forceinline__ bool wait_count(const volatile int* cnt, int target, const CtaAbort& ab, int where) {
  if (*cnt >= target) return true;
  const long long t0 = clock64();
  while (true) {
    if (*cnt >= target) return true;
    if (*ab.flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      raise_timeout(ab, where);
      return false;
    }
  }
}

// Launch order with L2 locality.  Blocks are grouped by heads: a group holds
// `group` consecutive heads and all of their `tiles` tiles, so the blocks that
// share a head's K/V (forward) or Q/dO (backward) run at the same time and read
// them from L2.  Inside a group, tile rank 0 (the heaviest under the causal
// mask) comes first and the head varies fastest.
__device__ __forceinline__ void grouped_order(int L, int tiles, int BH, int group, int& tile, int& bh) {
  const int per_group = group * tiles;
  const int g0 = (L / per_group) * group;
  const int r = L % per_group;
  const int gsize = min(group, BH - g0);
  tile = r / gsize;
  bh = g0 + r % gsize;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace fa
