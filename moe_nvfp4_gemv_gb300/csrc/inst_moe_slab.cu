// Instantiations of the slab kernel's MoE modes: gate_up (routed chunks of up
// to kSlabChunk pairs of one expert and the shared expert's token chunks, H
// split over a cluster) and down_combine (chunks of up to 8 pairs, several
// row tiles per CTA over one resident activation slab).
#include "k_gemv_slab.cuh"
#include "launch.h"

namespace fp4 {

cudaError_t launch_slab_moe(int mode, const GemvParams& p, const LaunchCfg& cfg) {
  if (p.cw != kSlabMaxCW) return cudaErrorInvalidValue;  // 128-row tiles
  static int configured_up[64], configured_down[64];     // per device (0 = not yet)
  if (mode == kMoeGateUp) {
    cudaError_t e = configure_kernel(gemv_slab_kernel<2, kMoeGateUp>, configured_up, cfg.smem, cfg.cluster);
    if (e != cudaSuccess) return e;
    return launch_kernel(gemv_slab_kernel<2, kMoeGateUp>, (p.cw + 1) * 32, p, cfg);
  }
  if (mode == kMoeDown) {
    if (cfg.cluster != 1 || p.tiles_per_cta < 1) return cudaErrorInvalidValue;
    cudaError_t e = configure_kernel(gemv_slab_kernel<2, kMoeDown>, configured_down, cfg.smem, cfg.cluster);
    if (e != cudaSuccess) return e;
    return launch_kernel(gemv_slab_kernel<2, kMoeDown>, (p.cw + 1) * 32, p, cfg);
  }
  return cudaErrorInvalidValue;
}

cudaError_t slab_moe_regs(int mode, int* regs) {
  cudaFuncAttributes a;
  cudaError_t e = mode == kMoeGateUp   ? cudaFuncGetAttributes(&a, gemv_slab_kernel<2, kMoeGateUp>)
                  : mode == kMoeDown ? cudaFuncGetAttributes(&a, gemv_slab_kernel<2, kMoeDown>)
                                     : cudaErrorInvalidValue;
  if (e == cudaSuccess) *regs = a.numRegs;
  return e;
}

}  // namespace fp4
