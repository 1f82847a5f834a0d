// Instantiations of the dense NVFP4 GEMV (plain and silu_mul tiles share them).
#include "launch.h"

namespace fp4 {

cudaError_t launch_dense_fp4(int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
  switch (nt) {
    case 16: return run_gemv<kDenseFp4, 16>(p, cfg, info);
    case 32: return run_gemv<kDenseFp4, 32>(p, cfg, info);
    case 64: return run_gemv<kDenseFp4, 64>(p, cfg, info);
    case 128: return run_gemv<kDenseFp4, 128>(p, cfg, info);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fp4
