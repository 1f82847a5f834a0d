// Launchers of the W4A4 path's activation kernels: quantisation (bf16 ->
// NVFP4 codes and 128x4 scales, optionally the exact dequantised bf16) and
// the dequantisation of NVFP4 activations for the GEMM.
#include "k_quantize_act.cuh"
#include "launch.h"

namespace fp4 {

// CTAs for `items` threads' work, at most `per_sm` resident CTAs per SM
// (the grid-stride loops then start every CTA at once).
static cudaError_t grid_for(uint64_t items, int per_sm, unsigned* ctas) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  uint64_t n = (items + kQuantThreads - 1) / kQuantThreads;
  const uint64_t cap = static_cast<uint64_t>(sms) * per_sm;
  if (n > cap) n = cap;
  *ctas = static_cast<unsigned>(n < 1 ? 1 : n);
  return cudaSuccess;
}

cudaError_t launch_quantize_act(const void* x, int64_t ldx, const float* gsi, uint8_t* q, uint8_t* sf, void* x_deq,
                                int M, int K, int pdl, cudaStream_t stream) {
  const uint32_t kbp = static_cast<uint32_t>(((K / 16) + 3) / 4 * 4);
  const uint64_t npos = static_cast<uint64_t>((M + 127) / 128 * 128) * kbp;
  if (npos >= (1ull << 31)) return cudaErrorInvalidValue;  // (32-bit positions)
  unsigned ctas = 0;
  // one thread per position up to four 256-thread CTAs per SM (57 registers);
  // past that the grid-stride loop takes two positions per iteration
  cudaError_t e = grid_for(npos, 4, &ctas);
  if (e != cudaSuccess) return e;
  // with pdl, launched early (programmatic stream serialisation): the kernel
  // waits for the previous grid before it reads anything
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(ctas, 1, 1);
  lc.blockDim = dim3(kQuantThreads, 1, 1);
  lc.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = &attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, quantize_act_kernel, static_cast<const uint16_t*>(x), ldx, gsi, q, sf,
                            static_cast<uint16_t*>(x_deq), M, K, kbp, static_cast<uint32_t>(npos));
}

cudaError_t launch_dequantize_act(const uint8_t* q, const uint8_t* sf, void* x_deq, int M, int K,
                                  cudaStream_t stream) {
  const uint32_t kbp = static_cast<uint32_t>(((K / 16) + 3) / 4 * 4);
  const uint64_t nblk = static_cast<uint64_t>(M) * (K / 16);
  if (nblk >= (1ull << 31)) return cudaErrorInvalidValue;  // (32-bit positions)
  unsigned ctas = 0;
  cudaError_t e = grid_for(nblk, 8, &ctas);
  if (e != cudaSuccess) return e;
  dequantize_act_kernel<<<ctas, kQuantThreads, 0, stream>>>(q, sf, static_cast<uint16_t*>(x_deq), K, kbp,
                                                           static_cast<uint32_t>(nblk));
  return cudaGetLastError();
}

}  // namespace fp4
