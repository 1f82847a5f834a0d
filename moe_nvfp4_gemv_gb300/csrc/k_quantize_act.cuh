// k_quantize_act.cuh -- NVFP4 quantisation of bf16 activations for the W4A4
// path (vllm.model_executor.kernels.linear.nvfp4.flashinfer, the W4A4
// kernels' apply_weights: scaled_fp4_quant(x, input_global_scale_inv), then
// the NVFP4 x NVFP4 GEMM with alpha).
//
// The pages name the operation but not its arithmetic.  Reading: the output
// is an NVFP4 tensor of the weights' own format (E2M1 codes, element 2j in
// the low nibble of byte j; E4M3 block scales, one per 16 values, in the
// 128x4 layout) whose values e2m1 x e4m3 approximate x * gsi.  Per row m and
// 16-value block b, in binary32, each operation rounded to nearest even and
// none fused:
//   amax = max |x|;  s = (amax / 6) * gsi;  sf = E4M3(s) (nearest, ties to
//   even, saturating at 448);  r = gsi / e4m3(sf) (0 if the scale is 0);
//   code = E2M1(x * r) (nearest, ties to the even code, saturating at 6; a
//   value that rounds to zero is stored as +0).
//
// HBM-bound: one thread per position (row r, block kb) of the padded scale
// layout, roundup(M, 128) x roundup(K / 16, 4) positions, kb fastest, so a
// warp's activation loads (32 bytes each) and code stores (8 bytes each)
// are contiguous; positions in the padding write a zero scale byte only.
// The E2M1 and E4M3 roundings are the conversion instructions' (round to
// nearest even, saturating to the largest finite value), the divisions
// IEEE-rounded (__fdiv_rn), the products __fmul_rn (no contraction).
// Optionally the exact dequantised values e2m1 x e4m3 (bf16, no global
// scale) go to x_deq, the operand of the W4A4 GEMM.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace fp4 {

constexpr int kQuantThreads = 256;

// Eight floats -> eight E2M1 codes (element i in nibble i) with the
// conversion instruction (round to nearest even, saturating at 6), then
// every zero magnitude stored as +0: a nibble's magnitude plus 7 sets its bit
// 3 exactly when the magnitude is not zero (no carry leaves the nibble).
__device__ __forceinline__ uint32_t e2m1x8_codes(const float* v) {
  uint32_t w;
  asm("{ .reg .b8 t0, t1, t2, t3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3}; }"
      : "=r"(w)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  const uint32_t nz = ((w & 0x77777777u) + 0x77777777u) & 0x88888888u;
  return w & (0x77777777u | nz);
}

// E2M1 code -> value (exact in float).
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t m = c & 7u;  // 0, 0.5 (subnormal), then 2^(m / 2 - 1) x (1 or 1.5)
  const float mag = m < 2u ? 0.5f * static_cast<float>(m)
                           : static_cast<float>(1u << (m / 2u - 1u)) * ((m & 1u) ? 1.5f : 1.0f);
  return (c & 8u) ? -mag : mag;
}

// Nearest finite E4M3 byte of s >= 0 (round to nearest even, saturating).
__device__ __forceinline__ uint32_t e4m3_code(float s) {
  unsigned short d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(d) : "f"(s));
  return d & 0xFFu;
}

__device__ __forceinline__ float e4m3_value(uint32_t b) {
  unsigned int h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<unsigned short>(b & 0xFFu)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}

__global__ void __launch_bounds__(kQuantThreads) quantize_act_kernel(const uint16_t* __restrict__ x, int64_t ldx,
                                                                    const float* __restrict__ gsi_p,
                                                                    uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                                    uint16_t* __restrict__ x_deq, int M, int K,
                                                                    uint32_t kbp, uint32_t npos) {
  // (the GEMM launched after this grid may start now and stream its weights;
  // it reads this grid's outputs only after waiting for the grid to end)
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();  // x (and gsi) may come from the previous grid
  const float gsi = __ldg(gsi_p);
  const uint32_t kb_used = static_cast<uint32_t>(K / 16);
  auto quant_block = [&](uint32_t r, uint32_t kb, uint32_t soff, const uint4& a, const uint4& b) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float v[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      amax = fmaxf(amax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
    }
    const float s = __fmul_rn(__fdiv_rn(amax, 6.0f), gsi);
    const uint32_t sc = e4m3_code(s);
    const float e = e4m3_value(sc);
    const float rcp = e > 0.0f ? __fdiv_rn(gsi, e) : 0.0f;
    float sv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) sv[i] = __fmul_rn(v[i], rcp);  // (rcp = 0: all +-0, codes 0)
    const uint32_t codes[2] = {e2m1x8_codes(sv), e2m1x8_codes(sv + 8)};
    *reinterpret_cast<uint2*>(q + static_cast<int64_t>(r) * (K / 2) + 8 * kb) = make_uint2(codes[0], codes[1]);
    sf[soff] = static_cast<uint8_t>(sc);
    if (x_deq) {
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float d0 = e2m1_value((codes[i / 4] >> (8 * (i % 4))) & 0xFu) * e;
        const float d1 = e2m1_value((codes[i / 4] >> (8 * (i % 4) + 4)) & 0xFu) * e;
        o[i] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(d0))) |
               (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(d1))) << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(x_deq + static_cast<int64_t>(r) * K + 16 * kb);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  };
  // two positions per thread and iteration, both loads issued first (64
  // bytes in flight per thread)
  const uint32_t stride = gridDim.x * kQuantThreads;
  for (uint32_t pos0 = blockIdx.x * kQuantThreads + threadIdx.x; pos0 < npos; pos0 += 2 * stride) {
    uint32_t r[2], kb[2], soff[2];
    bool live[2];
    uint4 a[2], b[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t pos = pos0 + u * stride;  // (< 2^31 + 2 stride: no wrap)
      r[u] = pos / kbp;
      kb[u] = pos - r[u] * kbp;
      soff[u] = ((r[u] >> 7) * (kbp >> 2) + (kb[u] >> 2)) * 512u + (r[u] & 31u) * 16u + ((r[u] & 127u) >> 5) * 4u +
                (kb[u] & 3u);
      live[u] = pos < npos && r[u] < static_cast<uint32_t>(M) && kb[u] < kb_used;
      if (live[u]) {
        const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(r[u]) * ldx + 16 * kb[u]);
        a[u] = __ldcs(src);
        b[u] = __ldcs(src + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (pos0 + u * stride >= npos) break;
      if (live[u]) quant_block(r[u], kb[u], soff[u], a[u], b[u]);
      else sf[soff[u]] = 0;  // padding of the 128x4 layout
    }
  }
}

// x_deq [M, K] bf16 = e2m1 x e4m3 of an NVFP4 activation tensor (exact; no
// global scale): the W4A4 GEMM's operand when its caller passes codes and
// scales.  One thread per 16-value block, kb fastest.
__global__ void __launch_bounds__(kQuantThreads) dequantize_act_kernel(const uint8_t* __restrict__ q,
                                                                      const uint8_t* __restrict__ sf,
                                                                      uint16_t* __restrict__ x_deq, int K,
                                                                      uint32_t kbp, uint32_t nblk) {
  const uint32_t kb_used = static_cast<uint32_t>(K / 16);
  if (threadIdx.x == 0) pdl_launch_dependents();
  for (uint32_t i = blockIdx.x * kQuantThreads + threadIdx.x; i < nblk; i += gridDim.x * kQuantThreads) {
    const uint32_t r = i / kb_used, kb = i - r * kb_used;
    const uint32_t soff = ((r >> 7) * (kbp >> 2) + (kb >> 2)) * 512u + (r & 31u) * 16u + ((r & 127u) >> 5) * 4u +
                          (kb & 3u);
    const float e = e4m3_value(__ldg(sf + soff));
    const uint2 c = __ldg(reinterpret_cast<const uint2*>(q + static_cast<int64_t>(r) * (K / 2) + 8 * kb));
    const uint32_t codes[2] = {c.x, c.y};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float d0 = e2m1_value((codes[j / 4] >> (8 * (j % 4))) & 0xFu) * e;
      const float d1 = e2m1_value((codes[j / 4] >> (8 * (j % 4) + 4)) & 0xFu) * e;
      o[j] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(d0))) |
             (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(d1))) << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(x_deq + static_cast<int64_t>(r) * K + 16 * kb);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace fp4
