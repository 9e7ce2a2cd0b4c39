// Instantiation of the LM-head + argmax GEMV (borrowed row-major BF16 head
// streamed through 2-D tensor-map copies).
#include "gemv_launch.cuh"

namespace dflash {
cudaError_t gemv_argmax(int nt, const GemvArgs& a, const ArgmaxParams& p, const LaunchCfg& lc) {
  return gemv_argmax_impl(nt, a, p, lc);
}
}  // namespace dflash
