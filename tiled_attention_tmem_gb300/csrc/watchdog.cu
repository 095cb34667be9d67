// Self-test of the in-kernel watchdog: one warp waits on an mbarrier phase that
// nothing completes.  The bounded wait gives up after kWaitLimitCycles and
// records a timeout in the library's device error word, exactly as an expired
// wait inside the attention kernels would; the kernel then returns normally, so
// the context stays usable.
#include "common.cuh"
#include "fa.h"
#include "host.h"

namespace fa {

__global__ void __launch_bounds__(32, 1) watchdog_selftest_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  const CtaAbort ab{&abort_flag, err};
  // No thread arrives on the barrier: phase 0 never completes.
  (void)wait_warp(smem_u32(&bar), 0, ab, (kKSelfTest << 8) | 1);
}

fa_status launch_watchdog_selftest(int* err, cudaStream_t st) {
  watchdog_selftest_kernel<<<1, 32, 0, st>>>(err);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FA_OK : record_cuda_error(e);
}

}  // namespace fa

extern "C" fa_status fa_watchdog_selftest(void* stream) {
  int* err = fa::device_error_word();
  if (!err) return fa::record_cuda_error(cudaErrorMemoryAllocation);
  return fa::launch_watchdog_selftest(err, static_cast<cudaStream_t>(stream));
}
