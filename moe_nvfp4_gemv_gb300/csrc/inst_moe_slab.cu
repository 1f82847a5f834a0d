// Instantiation of the slab kernel's MoE gate_up mode (routed chunks of up to
// kSlabChunk pairs of one expert and the shared expert's token chunks, the
// CTA's activations resident in shared memory, K split over a cluster).
#include "k_gemv_slab.cuh"
#include "launch.h"

namespace fp4 {

cudaError_t launch_slab_moe(const GemvParams& p, const LaunchCfg& cfg) {
  if (p.cw != kSlabMaxCW) return cudaErrorInvalidValue;  // 128-row tiles: one [up; gate] group
  static int configured_smem[64];  // per device (0 = not yet)
  cudaError_t e = configure_kernel(gemv_slab_kernel<2, kMoeGateUp>, configured_smem, cfg.smem, cfg.cluster);
  if (e != cudaSuccess) return e;
  return launch_kernel(gemv_slab_kernel<2, kMoeGateUp>, (p.cw + 1) * 32, p, cfg);
}

cudaError_t slab_moe_regs(int* regs) {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, gemv_slab_kernel<2, kMoeGateUp>);
  if (e == cudaSuccess) *regs = a.numRegs;
  return e;
}

}  // namespace fp4
