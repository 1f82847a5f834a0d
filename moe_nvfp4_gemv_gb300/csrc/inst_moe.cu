// Instantiations of the MoE kernels: gate_up and down_combine.
#include "launch.h"

namespace fp4 {

cudaError_t launch_moe(int mode, int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
  if (mode == kMoeGateUp && nt == 16) return run_gemv<kMoeGateUp, 16>(p, cfg, info);
  if (mode == kMoeGateUp && nt == 32) return run_gemv<kMoeGateUp, 32>(p, cfg, info);
  if (mode == kMoeDown && nt == 16) return run_gemv<kMoeDown, 16>(p, cfg, info);
  if (mode == kMoeDown && nt == 32) return run_gemv<kMoeDown, 32>(p, cfg, info);
  return cudaErrorInvalidValue;
}

}  // namespace fp4
