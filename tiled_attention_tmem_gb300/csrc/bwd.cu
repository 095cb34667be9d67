// Backward launchers (placeholder until the backward kernels land).
#include "host.h"

namespace fa {
fa_status run_bwd(const void*, const void*, const void*, const void*, const void*, const float*,
                  void*, void*, void*, int, int, int, float, int, int, void*, cudaStream_t) {
  return FA_ERR_UNSUPPORTED;
}
bool bwd_supported(int, int) { return false; }
int bwd_launch_count(int, int) { return 0; }
}  // namespace fa
