// Instantiation of the GEMV launchers for the bf16 backbone weight type.
#include "gemv_launch.cuh"

namespace dflash {
template cudaError_t gemv_store<WT_BF16>(int, const GemvArgs&, const EpiStore&, const LaunchCfg&);
template cudaError_t gemv_resid<WT_BF16>(int, const GemvArgs&, const EpiResid&, const LaunchCfg&);
template cudaError_t gemv_swiglu<WT_BF16>(int, const GemvArgs&, void*, const LaunchCfg&);
template cudaError_t gemv_heads<WT_BF16>(int, const GemvArgs&, const EpiHeads&, const LaunchCfg&);
}  // namespace dflash
