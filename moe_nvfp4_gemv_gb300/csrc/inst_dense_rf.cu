// Instantiations of the register-fed dense NVFP4 GEMV (M <= 16).
#include "k_gemv_rf.cuh"
#include "launch.h"

namespace fp4 {

template <int kNT>
cudaError_t run_gemv_rf(const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
  using C = RfCfg<kNT>;
  if (info) {
    info->threads = C::kThreads;
    info->stage_bytes = C::kStageBytes;
    info->red_bytes = 0;
    info->inbox_bytes = C::kInboxBytes;
    info->tmem_cols = 0;
    return cudaSuccess;
  }
  auto k = gemv_rf_kernel<kNT>;
  static int configured_smem[64];  // per device (0 = not yet)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured_smem[dev] < static_cast<int>(cfg.smem)) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(cfg.smem));
    if (e != cudaSuccess) return e;
    if (cfg.cluster > 8) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    configured_smem[dev] = static_cast<int>(cfg.smem);
  }
  return launch_kernel(k, C::kThreads, p, cfg);
}

cudaError_t launch_dense_rf(int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
  switch (nt) {
    case 8: return run_gemv_rf<8>(p, cfg, info);
    case 16: return run_gemv_rf<16>(p, cfg, info);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fp4
