// launch.h -- host-side interface between the C API translation unit and the
// kernel translation units (each instantiates part of the kernel templates so
// the library compiles in parallel).
#pragma once

#include <cuda_runtime.h>

#include "k_gemv.cuh"

namespace fp4 {

struct LaunchCfg {
  dim3 grid;
  unsigned cluster;     // CTAs per cluster along x (1: no cluster)
  size_t smem;          // dynamic shared memory bytes
  int pdl;              // programmatic dependent launch
  cudaStream_t stream;
};

struct KernelInfo {
  int threads;
  int stage_bytes;    // tcgen05 BF16 / register-fed: ring stage; tcgen05 NVFP4: unused
  int x_slice_bytes;  // tcgen05 NVFP4: one activation slot
  int tmem_slots;     // tcgen05 NVFP4: tensor-memory A slots
  int red_bytes;
  int inbox_bytes;
  int tmem_cols;
};

// Per (mode, kNT) kernel: static facts (info != nullptr) or a launch.  Each
// returns cudaErrorInvalidValue for a combination that is not instantiated.
cudaError_t launch_dense_fp4(int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info);
// Register-fed NVFP4 kernel (k_gemv_rf.cuh): mode kDenseFp4, kMoeGateUp or
// kMoeDown, nt = 8 or 16.
cudaError_t launch_rf(int mode, int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info);
// The same kernel budgeted for three CTAs per SM (instantiated for kMoeDown, nt = 8).
cudaError_t launch_rf_occ3(int mode, int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info);
// The dense 8-token variant whose consumers convert the activations of 3 .. 8 tokens to f16.
cudaError_t launch_rf_coop(int mode, int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info);
// Clusters of `cluster` CTAs of the dense register-fed kernel that fit on the
// GPU at once with `smem` bytes of dynamic shared memory each.
cudaError_t rf_max_clusters(int mode, int nt, unsigned cluster, size_t smem, int* n);
// Slab kernel (k_gemv_slab.cuh): dense NVFP4, 1 .. 8 tokens, r = 16-row
// blocks per consumer warp (1 or 2); the block is (p.cw + 1) warps.
cudaError_t launch_slab(int r, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info);
// The slab kernel's MoE modes, kMoeGateUp or kMoeDown (r = 2, four consumer
// warps; down_combine without a cluster).
cudaError_t launch_slab_moe(int mode, const GemvParams& p, const LaunchCfg& cfg);
cudaError_t slab_moe_regs(int mode, int* regs);
// The combine of down_combine after the slab kernel (128-thread blocks; with
// cfg.pdl it waits for the slab kernel's grid before reading its y rows).
cudaError_t launch_moe_combine(const GemvParams& p, const LaunchCfg& cfg);
cudaError_t launch_moe_down_persist(const GemvParams& p, const LaunchCfg& cfg);
cudaError_t launch_quantize_act(const void* x, int64_t ldx, const float* gsi, uint8_t* q, uint8_t* sf, void* x_deq,
                                int M, int K, int pdl, cudaStream_t stream);
cudaError_t launch_dequantize_act(const uint8_t* q, const uint8_t* sf, void* x_deq, int M, int K,
                                  cudaStream_t stream);
// Clusters of `cluster` slab-kernel CTAs (cw consumer warps, `smem` bytes of
// dynamic shared memory) that fit on the GPU at once.
cudaError_t slab_max_clusters(int r, int cw, unsigned cluster, size_t smem, int* n);
// Registers per thread of the slab kernel with r row blocks per warp.
cudaError_t slab_regs(int r, int* regs);
cudaError_t launch_dense_bf16(int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info);
cudaError_t launch_moe(int mode, int nt, const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info);
// kbp: 16-wide K blocks per 128-row scale group in sf (0: roundup(K / 16, 4)).
cudaError_t launch_dequantize_rows(const uint8_t* w, const uint8_t* sf, void* out, int rows, int K, int kbp,
                                   cudaStream_t stream);

// Raises a kernel's dynamic shared-memory limit to `smem` (once per device
// and size; `configured` holds the size set per device) and allows
// clusters of more than 8 CTAs when asked for.
template <typename Kernel>
cudaError_t configure_kernel(Kernel k, int (&configured)[64], size_t smem, unsigned cluster) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev] < static_cast<int>(smem)) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured[dev] = static_cast<int>(smem);
  }
  if (cluster > 8) return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return cudaSuccess;
}

// Shared launch helper for the kernel translation units.
template <typename Kernel>
cudaError_t launch_kernel(Kernel kernel, int threads, const GemvParams& p, const LaunchCfg& cfg) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = cfg.grid;
  lc.blockDim = dim3(threads, 1, 1);
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = cfg.stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (cfg.cluster > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = cfg.cluster;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  if (cfg.pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  lc.attrs = attrs;
  lc.numAttrs = na;
  return cudaLaunchKernelEx(&lc, kernel, p);
}

template <int kMode, int kNT>
cudaError_t run_gemv(const GemvParams& p, const LaunchCfg& cfg, KernelInfo* info) {
  using C = Cfg<kMode, kNT>;
  if (info) {
    info->threads = C::kThreads;
    info->stage_bytes = C::kStageBytes;
    info->x_slice_bytes = C::kXSliceBytes;
    info->tmem_slots = C::kSlots;
    info->red_bytes = C::kRedBytes;
    info->inbox_bytes = C::kInboxBytes;
    info->tmem_cols = C::kTmemCols;
    return cudaSuccess;
  }
  auto k = gemv_kernel<kMode, kNT>;
  static int configured_smem[64];  // per instantiation and device (0 = not yet)
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

}  // namespace fp4
