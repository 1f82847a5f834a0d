// dequant.cuh -- exact NVFP4 -> bf16 dequantization in registers.
//
// An E2M1 code c = (s, e1, e0, m) placed in bf16 bits as
//     bit 15 = s, bits 8..6 = (e1, e0, m)
// is the bf16 number e2m1(c) * 2^-126 (for e = 0 the pattern is the bf16
// subnormal 0.m * 2^-126, which is again e2m1(c) * 2^-126).  One bf16x2
// multiply by a block scale s' = e4m3 * 2^(126-kShift) then yields
//     e2m1(c) * e4m3 * 2^-kShift,
// an exact bf16 value (<= 6 significant bits, far from over/underflow).
// The GEMV keeps the 2^-kShift factor (kShift = 8 keeps s' below the bf16
// maximum for every finite e4m3) and multiplies the fp32 accumulator by
// 2^kShift at the end, which is exact.
//
// Bit placement needs only a shift per field when the two codes of a bf16x2
// pair sit 16 bits apart in the source word, so a 32-bit word of 8 codes
// (K order c0..c7) yields the pairs (c0,c4), (c2,c6), (c1,c5), (c3,c7).  The
// GEMV applies the same permutation to the activations' K order inside every
// aligned group of 8 (see perm_x8); dequantize_rows undoes it with byte
// permutes.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace fp4 {

constexpr int kShift = 8;

// 8 codes -> 4 bf16x2 words of raw values (times 2^-126), permuted pairs
// r[0] = (c0, c4), r[1] = (c2, c6), r[2] = (c1, c5), r[3] = (c3, c7).
__device__ __forceinline__ void e2m1x8_raw_perm(uint32_t w, uint32_t (&r)[4]) {
  const uint32_t kMag = 0x01C001C0u;  // bf16 bits 8..6 of both halves
  const uint32_t ws_even = w & 0x08080808u;  // sign bits of c0, c2, c4, c6
  const uint32_t ws_odd = w & 0x80808080u;   // sign bits of c1, c3, c5, c7
  // lop3 0xD8 = c ? b : a  (a: sign source, b: magnitude source, c: kMag)
  asm("lop3.b32 %0, %1, %2, %3, 0xD8;" : "=r"(r[0]) : "r"(ws_even << 12), "r"(w << 6), "r"(kMag));
  asm("lop3.b32 %0, %1, %2, %3, 0xD8;" : "=r"(r[1]) : "r"(ws_even << 4), "r"(w >> 2), "r"(kMag));
  asm("lop3.b32 %0, %1, %2, %3, 0xD8;" : "=r"(r[2]) : "r"(ws_odd << 8), "r"(w << 2), "r"(kMag));
  asm("lop3.b32 %0, %1, %2, %3, 0xD8;" : "=r"(r[3]) : "r"(ws_odd), "r"(w >> 6), "r"(kMag));
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Two e4m3 scale bytes (low byte first) -> two replicated bf16x2 multipliers
// s' = e4m3 * 2^(126 - kShift): lo for the first byte, hi for the second.
__device__ __forceinline__ void scale_pair_to_bf16x2(uint32_t two_bytes, uint32_t& lo, uint32_t& hi) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<unsigned short>(two_bytes & 0xFFFFu)));
  const float f0 = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu))) * 0x1p118f;
  const float f1 = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16))) * 0x1p118f;
  // Both products are exact with <= 4 significant bits, so the upper half of
  // the fp32 pattern is the exact bf16.
  lo = prmt(__float_as_uint(f0), 0u, 0x3232u);
  hi = prmt(__float_as_uint(f1), 0u, 0x3232u);
}

// 32 consecutive codes (16 bytes, K order) with the two scales of their 16-
// blocks -> 16 bf16x2 words of e2m1 * e4m3 * 2^-kShift, permuted within each
// group of 8 as e2m1x8_raw_perm.
__device__ __forceinline__ void dequant32_perm(const uint4& q, uint32_t s_lo, uint32_t s_hi, uint32_t (&out)[16]) {
  uint32_t r[4];
  e2m1x8_raw_perm(q.x, r);
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = bf16x2_mul(r[i], s_lo);
  e2m1x8_raw_perm(q.y, r);
#pragma unroll
  for (int i = 0; i < 4; ++i) out[4 + i] = bf16x2_mul(r[i], s_lo);
  e2m1x8_raw_perm(q.z, r);
#pragma unroll
  for (int i = 0; i < 4; ++i) out[8 + i] = bf16x2_mul(r[i], s_hi);
  e2m1x8_raw_perm(q.w, r);
#pragma unroll
  for (int i = 0; i < 4; ++i) out[12 + i] = bf16x2_mul(r[i], s_hi);
}

// Permutation of 8 consecutive bf16 K elements (one 16-byte chunk) into the
// order the permuted weight pairs use: [k0, k4, k2, k6, k1, k5, k3, k7].
__device__ __forceinline__ uint4 perm_x8(const uint4& v) {
  // v.x = (k0,k1), v.y = (k2,k3), v.z = (k4,k5), v.w = (k6,k7)
  uint4 o;
  o.x = prmt(v.x, v.z, 0x5410u);  // (k0, k4)
  o.y = prmt(v.y, v.w, 0x5410u);  // (k2, k6)
  o.z = prmt(v.x, v.z, 0x7632u);  // (k1, k5)
  o.w = prmt(v.y, v.w, 0x7632u);  // (k3, k7)
  return o;
}

// Inverse of the pair permutation for 4 words from e2m1x8_raw_perm-ordered
// results back to natural K order (k0,k1), (k2,k3), (k4,k5), (k6,k7).
__device__ __forceinline__ void unperm4(const uint32_t (&p)[4], uint32_t (&o)[4]) {
  o[0] = prmt(p[0], p[2], 0x5410u);
  o[1] = prmt(p[1], p[3], 0x5410u);
  o[2] = prmt(p[0], p[2], 0x7632u);
  o[3] = prmt(p[1], p[3], 0x7632u);
}

// --- f16 route --------------------------------------------------------------
// cvt.rn.f16x2.e2m1x2 turns one code byte (two codes, K order) into an exact
// f16 pair, and an e2m1 value times an e4m3 scale (<= 6 significant bits,
// magnitude in [2^-10, 2688]) is again an exact normal f16.  So 8 codes cost
// 4 conversions and 4 f16x2 multiplies, about half of the bf16 route above,
// and the pairs stay in natural K order.  The activations then have to be
// f16 as well (one MMA type per instruction); callers convert them and fall
// back to the bf16 route where a value is not exactly representable.

// 8 codes (natural K order) times a replicated f16x2 scale -> 4 f16x2 words
// (k0,k1) (k2,k3) (k4,k5) (k6,k7).
__device__ __forceinline__ void dequant8_f16(uint32_t w, uint32_t s2, uint32_t (&r)[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
#pragma unroll
  for (int i = 0; i < 4; ++i) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r[i]) : "r"(r[i]), "r"(s2));
}

// Two e4m3 scale bytes (low byte first) -> replicated f16x2 scales.
__device__ __forceinline__ void scale_pair_to_f16x2(uint32_t two_bytes, uint32_t& lo, uint32_t& hi) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<unsigned short>(two_bytes & 0xFFFFu)));
  lo = prmt(h, h, 0x1010u);
  hi = prmt(h, h, 0x3232u);
}

// The same scales times a replicated f16x2 `mul` (a power of two that keeps
// every product exact, see the slab kernel's shifted f16 route).
__device__ __forceinline__ void scale_pair_to_f16x2_scaled(uint32_t two_bytes, uint32_t mul, uint32_t& lo,
                                                           uint32_t& hi) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<unsigned short>(two_bytes & 0xFFFFu)));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(h) : "r"(h), "r"(mul));
  lo = prmt(h, h, 0x1010u);
  hi = prmt(h, h, 0x3232u);
}

// bf16 pair -> f16 pair; false if either value is not exactly representable
// in f16 (too large, too small for its bits, or NaN).
__device__ __forceinline__ bool bf16x2_to_f16x2_exact(uint32_t v, uint32_t& out) {
  const float lo = __uint_as_float(v << 16);
  const float hi = __uint_as_float(v & 0xFFFF0000u);
  uint32_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
  out = h;
  const float blo = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
  const float bhi = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
  return (blo == lo) & (bhi == hi);
}

}  // namespace fp4
