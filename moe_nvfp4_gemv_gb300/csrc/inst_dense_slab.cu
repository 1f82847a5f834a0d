// Instantiations of the slab kernel (dense NVFP4 GEMV, 1 .. 8 tokens, the
// CTA's activations resident in shared memory).
#include "k_gemv_slab.cuh"
#include "launch.h"

namespace fp4 {

template <int kR>
cudaError_t configure_slab(size_t smem, unsigned cluster) {
  static int configured_smem[64];  // per device (0 = not yet)
  return configure_kernel(gemv_slab_kernel<kR>, configured_smem, smem, cluster);
}

cudaError_t launch_slab(int r, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
  if (r != 1 && r != 2) return cudaErrorInvalidValue;
  if (info) {
    info->threads = kSlabThreads;
    info->stage_bytes = 0;
    info->red_bytes = 0;
    info->inbox_bytes = SlabCfg<2>::kInboxFloats * 4;  // (the larger of the two)
    info->tmem_cols = 0;
    return cudaSuccess;
  }
  // (cw + 1) warps: cw consumers and the producer
  const int threads = (p.cw + 1) * 32;
  if (p.cw < 1 || p.cw > kSlabMaxCW) return cudaErrorInvalidValue;
  cudaError_t e = r == 1 ? configure_slab<1>(cfg.smem, cfg.cluster) : configure_slab<2>(cfg.smem, cfg.cluster);
  if (e != cudaSuccess) return e;
  return r == 1 ? launch_kernel(gemv_slab_kernel<1>, threads, p, cfg) : launch_kernel(gemv_slab_kernel<2>, threads, p, cfg);
}

cudaError_t slab_regs(int r, int* regs) {
  if (r != 1 && r != 2) return cudaErrorInvalidValue;
  cudaFuncAttributes a;
  cudaError_t e = r == 1 ? cudaFuncGetAttributes(&a, gemv_slab_kernel<1>) : cudaFuncGetAttributes(&a, gemv_slab_kernel<2>);
  if (e == cudaSuccess) *regs = a.numRegs;
  return e;
}

cudaError_t slab_max_clusters(int r, int cw, unsigned cluster, size_t smem, int* n) {
  if (r != 1 && r != 2) return cudaErrorInvalidValue;
  cudaError_t e = r == 1 ? configure_slab<1>(smem, cluster) : configure_slab<2>(smem, cluster);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t c = {};
  c.gridDim = dim3(cluster, 1, 1);
  c.blockDim = dim3((cw + 1) * 32, 1, 1);
  c.dynamicSmemBytes = smem;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = cluster;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  c.attrs = a;
  c.numAttrs = 1;
  return r == 1 ? cudaOccupancyMaxActiveClusters(n, gemv_slab_kernel<1>, &c)
                : cudaOccupancyMaxActiveClusters(n, gemv_slab_kernel<2>, &c);
}

}  // namespace fp4
