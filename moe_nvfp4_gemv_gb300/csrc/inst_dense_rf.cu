// Instantiations of the register-fed NVFP4 kernel (dense GEMV and both MoE
// kernels, chunks of at most 16 tokens / pairs).
#include "k_gemv_rf.cuh"
#include "launch.h"

namespace fp4 {

template <int kMode, int kNT>
cudaError_t run_gemv_rf(const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
  using C = RfCfg<kNT>;
  if (info) {
    info->threads = C::kThreads;
    info->stage_bytes = C::kXBytes;  // the activations' share; the host adds weights and scale groups
    info->red_bytes = 0;
    info->inbox_bytes = C::kInboxFloats * 4 + (kMode == kDenseFp4 ? 0 : C::kWorkBytes);
    info->tmem_cols = 0;
    return cudaSuccess;
  }
  auto k = gemv_rf_kernel<kMode, kNT>;
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

cudaError_t launch_rf(int mode, int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
#define FP4_CASE(M_, NT_) \
  if (mode == M_ && nt == NT_) return run_gemv_rf<M_, NT_>(p, cfg, info);
  FP4_CASE(kDenseFp4, 8) FP4_CASE(kDenseFp4, 16)
  FP4_CASE(kMoeGateUp, 8) FP4_CASE(kMoeGateUp, 16)
  FP4_CASE(kMoeDown, 8) FP4_CASE(kMoeDown, 16)
#undef FP4_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fp4
