// Instantiation of the GEMV launchers for the q5_0 backbone weight type.
#include "gemv_launch.cuh"

namespace dflash {
template cudaError_t gemv_store<WT_Q5_0>(int, const GemvArgs&, const EpiStore&, const LaunchCfg&);
template cudaError_t gemv_resid<WT_Q5_0>(int, const GemvArgs&, const EpiResid&, const LaunchCfg&);
template cudaError_t gemv_swiglu<WT_Q5_0>(int, const GemvArgs&, void*, const LaunchCfg&);
template cudaError_t gemv_heads<WT_Q5_0>(int, const GemvArgs&, const EpiHeads&, const LaunchCfg&);
}  // namespace dflash
