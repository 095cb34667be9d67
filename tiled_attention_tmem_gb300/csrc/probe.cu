// Throughput probe of the exponential unit.  The issue thread "Potential
// algorithmic improvements for backward pass" argues that the exponential, not
// the matrix multiply, limits attention as tensor throughput grows, and prices
// it as an ex2 issue rate per SM per clock; the kernels here take every
// exponential with ex2.approx.ftz.f32, so this probe measures that
// instruction's rate on the running GPU.
#include "common.cuh"
#include "fa.h"
#include "host.h"

namespace fa {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeChains = 8;

// Each thread runs kProbeChains independent chains x <- 2^(-x) (the negation is
// an operand modifier of the instruction): from x in (0, 1] every value stays in
// [0.5, 1), so no denormal or special input occurs; the sum of the chains is
// written so that nothing is optimised away.
__global__ void __launch_bounds__(kProbeThreads) ex2_probe_kernel(float* sink, int iters) {
  float x[kProbeChains];
#pragma unroll
  for (int c = 0; c < kProbeChains; ++c) x[c] = 0.25f + 0.01f * (float)(c + (threadIdx.x & 7));
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kProbeChains; ++c) x[c] = ex2(-x[c]);
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kProbeChains; ++c) s += x[c];
  sink[(size_t)blockIdx.x * kProbeThreads + threadIdx.x] = s;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_ex2_probe(float* sink, int blocks, int iters, long long* count, void* stream) {
  if (count) *count = 0;
  if (!sink || blocks <= 0 || iters <= 0) return FA_ERR_INVALID_ARG;
  fa::ex2_probe_kernel<<<blocks, fa::kProbeThreads, 0, static_cast<cudaStream_t>(stream)>>>(sink, iters);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fa::record_cuda_error(e);
  if (count) *count = (long long)blocks * fa::kProbeThreads * fa::kProbeChains * iters;
  return FA_OK;
}
