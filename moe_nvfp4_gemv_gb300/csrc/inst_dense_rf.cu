// Instantiations of the register-fed NVFP4 kernel (dense GEMV and both MoE
// kernels, chunks of at most 16 tokens / pairs).
#include "k_gemv_rf.cuh"
#include "launch.h"

namespace fp4 {

// Raise the kernel's dynamic shared-memory limit to `smem` (once per device
// and size).
template <int kMode, int kNT, int kOcc = 2, bool kCoop = false>
cudaError_t configure_rf(size_t smem, unsigned cluster) {
  auto k = gemv_rf_kernel<kMode, kNT, kOcc, kCoop>;
  static int configured_smem[64];  // per device (0 = not yet)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured_smem[dev] < static_cast<int>(smem)) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured_smem[dev] = static_cast<int>(smem);
  }
  if (cluster > 8) return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return cudaSuccess;
}

template <int kMode, int kNT, int kOcc = 2, bool kCoop = false>
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
  cudaError_t e = configure_rf<kMode, kNT, kOcc, kCoop>(cfg.smem, cfg.cluster);
  if (e != cudaSuccess) return e;
  return launch_kernel(gemv_rf_kernel<kMode, kNT, kOcc, kCoop>, C::kThreads, p, cfg);
}

template <int kMode, int kNT, bool kCoop = false>
cudaError_t rf_clusters(unsigned cluster, size_t smem, int* n) {
  cudaError_t e = configure_rf<kMode, kNT, 2, kCoop>(smem, cluster);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t c = {};
  c.gridDim = dim3(cluster, 1, 1);
  c.blockDim = dim3(RfCfg<kNT>::kThreads, 1, 1);
  c.dynamicSmemBytes = smem;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = cluster;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  c.attrs = a;
  c.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, gemv_rf_kernel<kMode, kNT, 2, kCoop>, &c);
}

cudaError_t rf_max_clusters(int mode, int nt, unsigned cluster, size_t smem, int* n) {
#define FP4_CASE(M_, NT_) \
  if (mode == M_ && nt == NT_) return rf_clusters<M_, NT_>(cluster, smem, n);
  FP4_CASE(kDenseFp4, 8) FP4_CASE(kDenseFp4, 16)
#undef FP4_CASE
  return cudaErrorInvalidValue;
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

cudaError_t launch_rf_occ3(int mode, int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
  if (mode == kMoeDown && nt == 8) return run_gemv_rf<kMoeDown, 8, 3>(p, cfg, info);
  return cudaErrorInvalidValue;
}

cudaError_t launch_rf_coop(int mode, int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
  if (mode == kDenseFp4 && nt == 8) return run_gemv_rf<kDenseFp4, 8, 2, true>(p, cfg, info);
  if (mode == kDenseFp4 && nt == 16) return run_gemv_rf<kDenseFp4, 16, 2, true>(p, cfg, info);
  return cudaErrorInvalidValue;
}

}  // namespace fp4
