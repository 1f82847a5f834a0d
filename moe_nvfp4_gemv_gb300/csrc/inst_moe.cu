// Instantiations of the MoE kernels: gate_up (kT = 2) and down_combine (kT = 1).
#include "launch.h"

namespace fp4 {

cudaError_t launch_moe(int mode, int t, int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
  if (mode == kMoeGateUp && t == 2 && nt == 16) return run_gemv<kMoeGateUp, 2, 16>(p, cfg, info);
  if (mode == kMoeGateUp && t == 2 && nt == 32) return run_gemv<kMoeGateUp, 2, 32>(p, cfg, info);
  if (mode == kMoeDown && t == 1 && nt == 16) return run_gemv<kMoeDown, 1, 16>(p, cfg, info);
  if (mode == kMoeDown && t == 1 && nt == 32) return run_gemv<kMoeDown, 1, 32>(p, cfg, info);
  return cudaErrorInvalidValue;
}

}  // namespace fp4
