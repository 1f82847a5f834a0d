// Instantiations of the dense NVFP4 GEMV (kT = 1 plain, kT = 2 silu_mul).
#include "launch.h"

namespace fp4 {

cudaError_t launch_dense_fp4(int t, int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
#define FP4_CASE(T_, NT_) \
  if (t == T_ && nt == NT_) return run_gemv<kDenseFp4, T_, NT_>(p, cfg, info);
  FP4_CASE(1, 16) FP4_CASE(1, 32) FP4_CASE(1, 64) FP4_CASE(1, 128)
  FP4_CASE(2, 16) FP4_CASE(2, 32) FP4_CASE(2, 64) FP4_CASE(2, 128)
#undef FP4_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fp4
