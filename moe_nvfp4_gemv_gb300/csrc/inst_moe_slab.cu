// Instantiations of the slab kernel's MoE modes: gate_up (routed chunks of
// pairs of one expert and the shared expert's token chunks; split form: H
// split over a cluster; grouped form: several tiles per CTA over one
// resident activation slab) and down_combine (grouped, one CTA per item,
// and its persistent form), and the combine kernel that follows either.
#include "k_gemv_slab.cuh"
#include "k_moe_down_persist.cuh"
#include "launch.h"

namespace fp4 {

// down_combine after the slab kernel: one thread per 8 consecutive h of one
// token, grid-strided; waits for the previous grid (the slab kernel or its
// persistent form, whose y rows it reads) and skips the tiles a CTA of that
// grid tagged as given up.
__global__ void __launch_bounds__(128) moe_combine_kernel(const __grid_constant__ GemvParams p) {
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();
  const int per_token = p.n_out / 8;
  const unsigned long long tag = abort_tag(p.epoch);
  for (int it = blockIdx.x * blockDim.x + threadIdx.x; it < p.M * per_token; it += gridDim.x * blockDim.x) {
    const int t = it / per_token, h = 8 * (it % per_token);
    if (__ldcg(p.counters + h / 128) == tag) continue;
    moe_combine_item(p, t, h);
  }
}


cudaError_t launch_moe_combine(const GemvParams& p, const LaunchCfg& cfg) {
  return launch_kernel(moe_combine_kernel, 128, p, cfg);
}

cudaError_t launch_slab_moe(int mode, const GemvParams& p, const LaunchCfg& cfg) {
  if (p.cw != kSlabMaxCW) return cudaErrorInvalidValue;  // 128-row tiles
  static int configured_up[64], configured_grouped[64], configured_down[64];  // per device (0 = not yet)
  if (mode == kMoeGateUp && p.tiles_per_cta > 0) {  // the grouped form
    if (cfg.cluster != 1) return cudaErrorInvalidValue;
    cudaError_t e = configure_kernel(gemv_slab_kernel<2, kMoeGateUp, true>, configured_grouped, cfg.smem, 1);
    if (e != cudaSuccess) return e;
    return launch_kernel(gemv_slab_kernel<2, kMoeGateUp, true>, (p.cw + 1) * 32, p, cfg);
  }
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

cudaError_t launch_moe_down_persist(const GemvParams& p, const LaunchCfg& cfg) {
  if (p.cw != kSlabMaxCW || cfg.cluster != 1) return cudaErrorInvalidValue;
  static int configured[64];  // per device (0 = not yet)
  cudaError_t e = configure_kernel(moe_down_persist_kernel<2>, configured, cfg.smem, 1);
  if (e != cudaSuccess) return e;
  return launch_kernel(moe_down_persist_kernel<2>, (p.cw + 1) * 32, p, cfg);
}

// (gate_up, down_combine: the larger of their two forms)
cudaError_t slab_moe_regs(int mode, int* regs) {
  cudaFuncAttributes a, b;
  cudaError_t e = cudaErrorInvalidValue;
  if (mode == kMoeGateUp) {
    e = cudaFuncGetAttributes(&a, gemv_slab_kernel<2, kMoeGateUp>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&b, gemv_slab_kernel<2, kMoeGateUp, true>);
    if (e == cudaSuccess && b.numRegs > a.numRegs) a.numRegs = b.numRegs;
  } else if (mode == kMoeDown) {  // (the larger of the grid and the persistent form)
    e = cudaFuncGetAttributes(&a, gemv_slab_kernel<2, kMoeDown>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&b, moe_down_persist_kernel<2>);
    if (e == cudaSuccess && b.numRegs > a.numRegs) a.numRegs = b.numRegs;
  }
  if (e == cudaSuccess) *regs = a.numRegs;
  return e;
}

}  // namespace fp4
