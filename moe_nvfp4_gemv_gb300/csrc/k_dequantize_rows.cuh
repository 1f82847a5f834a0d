// k_dequantize_rows.cuh -- bf16 [rows, K] = e2m1 * e4m3 exactly
// (vllm.models.flint.ops.nvfp4_gemv, dequantize_rows).
//
// HBM-bound streaming kernel: per 32 weights it reads 16 bytes of codes and
// 2 scale bytes and writes 64 bytes.  The [rows, K/2] code matrix and the
// [rows, K] output are both contiguous, so the kernel walks them as one flat
// stream of 16-byte code chunks (chunk c -> row c / (K/32), K offset
// 32 * (c % (K/32))): loads and stores are fully coalesced, 128-bit wide.
// Scales are read through the read-only path from the 128x4 layout; one
// chunk needs the scales of two consecutive 16-blocks, which are adjacent
// bytes there.  A warp's 32 chunks are consecutive, so their outputs are one
// contiguous 2 KB block: each thread's 64 bytes go through shared memory and
// come back out as four warp-wide stores of 512 contiguous bytes (whole 32-byte
// sectors), instead of 16-byte stores that each half-fill 64 sectors.
#pragma once

#include "common.cuh"
#include "dequant.cuh"

namespace fp4 {

constexpr int kDqThreads = 256;
constexpr int kDqUnroll = 4;

__device__ __forceinline__ uint32_t scale_offset(uint32_t r, uint32_t kb, uint32_t kbp) {
  return ((r >> 7) * (kbp >> 2) + (kb >> 2)) * 512u + (r & 31u) * 16u + ((r & 127u) >> 5) * 4u + (kb & 3u);
}

__global__ void __launch_bounds__(kDqThreads) dequantize_rows_kernel(const uint4* __restrict__ w,
                                                                    const uint8_t* __restrict__ sf,
                                                                    uint4* __restrict__ out, uint64_t nchunks,
                                                                    uint32_t chunks_per_row, uint32_t kbp) {
  __shared__ __align__(16) uint4 stage[kDqThreads / 32][128];  // 2 KB per warp
  const int lane = threadIdx.x % 32;
  uint4* const ws = stage[threadIdx.x / 32];
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kDqThreads;
  uint64_t c = static_cast<uint64_t>(blockIdx.x) * kDqThreads + threadIdx.x;
  // (the warp iterates together: its __syncwarp()s need every lane; each
  // chunk is bounds-checked)
  for (; c - lane < nchunks; c += stride * kDqUnroll) {
    uint4 q[kDqUnroll];
    uint32_t s2[kDqUnroll];
#pragma unroll
    for (int u = 0; u < kDqUnroll; ++u) {
      const uint64_t cc = c + u * stride;
      if (cc < nchunks) {
        const uint32_t r = static_cast<uint32_t>(cc / chunks_per_row);
        const uint32_t kb = 2u * static_cast<uint32_t>(cc % chunks_per_row);
        q[u] = __ldcs(w + cc);
        s2[u] = __ldg(reinterpret_cast<const unsigned short*>(sf + scale_offset(r, kb, kbp)));
      }
    }
#pragma unroll
    for (int u = 0; u < kDqUnroll; ++u) {
      const uint64_t cc = c + u * stride;
      if (cc < nchunks) {
        uint32_t s_lo, s_hi;
        scale_pair_to_bf16x2(s2[u], s_lo, s_hi);
        const uint32_t words[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t r[4], p[4], o[4];
          e2m1x8_raw_perm(words[i], r);
          const uint32_t s = i < 2 ? s_lo : s_hi;
#pragma unroll
          for (int j = 0; j < 4; ++j) p[j] = bf16x2_mul(bf16x2_mul(r[j], s), 0x43804380u);  // * 2^kShift
          unperm4(p, o);
          // 16-byte piece 4 lane + i of the warp's block; the XOR spreads
          // a store instruction's 32 pieces over all banks
          ws[(4 * lane + i) ^ ((lane >> 1) & 3)] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      __syncwarp();
      // piece 32 i + lane of the warp's block, i.e. chunk 8 i + lane / 4 of
      // the warp, part lane % 4 (the warp's chunks are consecutive)
      const uint64_t wc0 = c - lane + u * stride;  // the warp's first chunk
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int piece = 32 * i + lane;
        const int owner = piece / 4;  // lane that produced it
        if (wc0 + owner < nchunks) out[wc0 * 4 + piece] = ws[piece ^ ((owner >> 1) & 3)];
      }
      __syncwarp();
    }
  }
}

}  // namespace fp4
