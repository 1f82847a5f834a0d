// dequantize_rows launcher.
#include "k_dequantize_rows.cuh"
#include "launch.h"

namespace fp4 {

cudaError_t launch_dequantize_rows(const uint8_t* w, const uint8_t* sf, void* out, int rows, int K, int kbp_in,
                                   cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const uint64_t nchunks = static_cast<uint64_t>(rows) * (K / 32);
  const uint64_t per_cta = static_cast<uint64_t>(kDqThreads) * kDqUnroll;
  uint64_t ctas = (nchunks + per_cta - 1) / per_cta;
  const uint64_t cap = static_cast<uint64_t>(sms) * 8;  // 8 x 256 threads per SM
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  const uint32_t kbp = kbp_in > 0 ? static_cast<uint32_t>(kbp_in) : ((K / 16) + 3) / 4 * 4;
  dequantize_rows_kernel<<<static_cast<unsigned>(ctas), kDqThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(w), sf, reinterpret_cast<uint4*>(out), nchunks, K / 32, kbp);
  return cudaGetLastError();
}

}  // namespace fp4
