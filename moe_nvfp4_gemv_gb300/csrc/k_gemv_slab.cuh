// k_gemv_slab.cuh -- the NVFP4 GEMV with the CTA's activations resident in
// shared memory: the dense GEMV for 1 .. 4 tokens on large weights, and the
// MoE pair (gate_up: split and grouped forms; down_combine: grouped, its
// combine a kernel of its own after the grid; beyond one wave of CTAs
// down_combine runs on the persistent form of this kernel,
// k_moe_down_persist.cuh).
//
// Same operations as the register-fed kernel k_gemv_rf.cuh
// (vllm.models.flint.ops.nvfp4_gemv, nvfp4_gemv, with or without silu_mul;
// vllm.models.flint.ops.moe_gemv, gate_up and down_combine), organised so
// that the only per-stage traffic is the weight stream:
//
//   * The CTA's activation slab, x[0 .. M)[k_begin .. k_end) (MoE: the rows
//     of its chunk of pairs of one expert), is read from global memory once,
//     after griddepcontrol.wait, by all consumer threads and kept in shared
//     memory for the whole launch (64-K atoms of M rows x 128 bytes, 16-byte
//     chunks XOR-swizzled by token).  A 256-K stage whose activations are
//     all exactly representable in f16 is converted to f16 in place (the f16
//     route: cvt.rn.f16x2.e2m1x2 on the weights, f16 MMAs); a stage whose
//     values fit f16's normal range after a power-of-two shift s takes the
//     same route with x 2^s and the scales times 2^-s (exact, the same
//     products); any other stage keeps its bf16 values and runs the bf16
//     bit-placement route (dequant.cuh).  The routes form exact products and
//     accumulate in fp32 (f16 route and bf16 route separately, summed at the
//     end).
//   * The ring holds only weights and their scale groups (TMA boxes and
//     bulk copies).  The producer warp never waits for the previous grid:
//     weights are not written by it, so the ring fills completely under PDL.
//   * No converter warp and no per-stage CTA barrier: a consumer warp waits
//     on one full barrier per stage and releases the stage with one arrival.
//   * The block has exactly cw consumer warps and the producer warp (the
//     host launches (cw + 1) x 32 threads), so no warp sits idle.
//   * Grouped MoE forms stream T row tiles per CTA in turn over the same
//     resident rows, the ring running across the tile boundary; each tile's
//     outputs are written from registers without a CTA barrier (gate_up
//     pairs each feature's up and gate rows in one thread).
//
// Fragment mapping as in k_gemv_rf.cuh: thread (g, c) of consumer warp w
// holds, for each of its kR 16-row blocks b, MMA rows g and g + 8 = tile rows
// 16 (kR w + b) + sigma(g) and + 8, sigma = (0 4 1 5 2 6 3 7) (gate_up's
// grouped form: 64 b + 16 w + sigma(g)); in 128-K half h of a stage it reads
// code chunk 4 h + c of both rows.  The K split over the S CTAs of a cluster
// and its reduction through distributed shared memory are those of the
// register-fed kernel.
#pragma once

#include <type_traits>

#include "k_gemv_rf.cuh"

namespace fp4 {

constexpr int kSlabR = 2;             // 16-row blocks per consumer warp
constexpr int kSlabThreads = kSlabMaxCW * 32 + 32;
constexpr int kSlabMinBlocks = 3;     // CTAs per SM the registers are budgeted for

template <int kR>
struct SlabCfg {
  static constexpr int kChains = kR == 1 ? 4 : 2;  // independent fp32 accumulators per row block
  static constexpr int kInboxFloats = kSlabNT * (16 * kSlabMaxCW * kR + 16);
  static_assert(kInboxFloats * 4 <= SlabInboxBytes, "inbox");
};

// Named barrier 1 over the first n threads (the consumer warps).
__device__ __forceinline__ void cons_sync(int n) { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }

// Eight bf16 values -> eight f16 values; false if any is not exact in f16.
__device__ __forceinline__ bool bf16x8_to_f16x8_exact(const uint4& v, uint4& o) {
  bool e = bf16x2_to_f16x2_exact(v.x, o.x);
  e &= bf16x2_to_f16x2_exact(v.y, o.y);
  e &= bf16x2_to_f16x2_exact(v.z, o.z);
  e &= bf16x2_to_f16x2_exact(v.w, o.w);
  return e;
}

// f16 route with a power-of-two shift (stages with a value that is not an
// exact f16 as it is).  A stage's activations x run on the
// f16 route as x 2^s (f16) against weights e2m1 * (e4m3 2^-s) (f16), whose
// products equal x * e2m1 * e4m3 exactly: x 2^s is exact in f16 when every
// nonzero x 2^s lies in f16's normal range (a bf16 has 8 significant bits,
// a normal f16 11), and e4m3 2^-s and e2m1 * e4m3 2^-s are multiples of
// 2^-24 below 2^12 for s <= 14 (every e4m3 value is a multiple of 2^-9).
// So the shift moves the exponent between the operands and the products,
// and the accumulator, are those of the unshifted route.
//
// Largest and smallest biased exponent fields of the nonzero values among
// eight bf16 values (zeros give 0 and 255; a bf16 subnormal gives 0).
__device__ __forceinline__ void bf16x8_exp_range(const uint4& v, int& emax, int& emin) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  emax = 0;
  emin = 255;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t a = (w[q] >> (16 * half)) & 0x7FFFu;
      const int e = static_cast<int>(a >> 7);
      emax = max(emax, e);
      emin = min(emin, a != 0u ? e : 255);
    }
  }
}

// The shift of a stage whose nonzero activations have biased exponent
// fields in [emin, emax]: the largest s <= 14 with every x 2^s below 2^16
// (x < 2^(emax - 126)) and at least 2^-14 (x >= 2^(emin - 127)), or -1 when
// there is none (Inf, NaN, bf16 subnormals, or a range wider than f16's):
// the stage takes the bf16 route.
__device__ __forceinline__ int f16_shift(int emax, int emin) {
  const int s = min(14, 142 - emax);
  return (s >= 0 && s >= 113 - emin) ? s : -1;
}

// Eight bf16 values times 2^s (mul = 2^s) -> eight f16 values, exact when s
// is the stage's f16_shift.
__device__ __forceinline__ uint4 bf16x8_to_f16x8_scaled(const uint4& v, float mul) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float lo = __uint_as_float(w[q] << 16) * mul;
    const float hi = __uint_as_float(w[q] & 0xFFFF0000u) * mul;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o[q]) : "f"(hi), "f"(lo));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Replicated f16x2 of 2^-s (0 <= s <= 14: a normal f16).
__device__ __forceinline__ uint32_t f16x2_pow2_neg(int s) {
  const uint32_t b = static_cast<uint32_t>(15 - s) << 10;
  return b | (b << 16);
}

// One 128-K half h of a 256-K stage for a consumer warp of the slab
// kernels (f16 route): thread (g, c) of the warp, its kR row blocks' code
// rows at w_off and scale bytes at sf_off in the stage at `st`, the stage's
// activations at `xs` (64-K atoms of M rows x 128 bytes, 16-byte chunks
// XOR-swizzled by row % 8, f16, times 2^s), the scales times 2^-s (kScaled;
// sdown: f16x2_pow2_neg(s)).  `cvalid` false (a chunk past the end of a ragged last
// stage) gives zero A registers: that chunk's scales were not copied and may
// hold anything.
template <int kR, int kChains, bool kScaled>
__device__ __forceinline__ void slab_half_f16(float (&acc)[kChains][kR][4], uint32_t st, uint32_t xs, int h,
                                              bool cvalid, int M, const uint32_t (&w_off)[kR][2],
                                              const uint32_t (&sf_off)[kR][2], uint32_t key, int g, int c,
                                              uint32_t sdown) {
  const int j = 4 * h + c;
  uint4 A[kR][2];
  uint32_t slo[kR][2], shi[kR][2];
  const uint32_t sc_off = (j / 2) * 512 + 2 * (j % 2);
#pragma unroll
  for (int b = 0; b < kR; ++b) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      A[b][hr] = lds128(st + w_off[b][hr] + ((static_cast<uint32_t>(j) ^ key) * 16));
      if constexpr (kScaled) scale_pair_to_f16x2_scaled(lds16(st + sf_off[b][hr] + sc_off), sdown, slo[b][hr], shi[b][hr]);
      else scale_pair_to_f16x2(lds16(st + sf_off[b][hr] + sc_off), slo[b][hr], shi[b][hr]);
      if (!cvalid) slo[b][hr] = shi[b][hr] = 0u;
    }
  }
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int kk = 32 * j + 8 * w;
    const uint32_t u = kk / 64, ch = (kk % 64) / 8;
    const uint4 xv = lds128_if(xs + (u * M + g) * 128 + ((ch ^ static_cast<uint32_t>(g)) * 16), g < M);
#pragma unroll
    for (int b = 0; b < kR; ++b) {
      const uint32_t w0 = w == 0 ? A[b][0].x : w == 1 ? A[b][0].y : w == 2 ? A[b][0].z : A[b][0].w;
      const uint32_t w1 = w == 0 ? A[b][1].x : w == 1 ? A[b][1].y : w == 2 ? A[b][1].z : A[b][1].w;
      uint32_t r0[4], r1[4];
      dequant8_f16(w0, w < 2 ? slo[b][0] : shi[b][0], r0);
      dequant8_f16(w1, w < 2 ? slo[b][1] : shi[b][1], r1);
      mma_f16_16816(acc[(2 * w) % kChains][b], r0[0], r1[0], r0[1], r1[1], xv.x, xv.y);
      mma_f16_16816(acc[(2 * w + 1) % kChains][b], r0[2], r1[2], r0[3], r1[3], xv.z, xv.w);
    }
  }
}

// The same half on the bf16 route (the stage's activations are bf16; they
// are permuted in registers to the weight pairs' K order); products times
// 2^-kShift into accb.
template <int kR>
__device__ __forceinline__ void slab_half_bf16(float (&accb)[kR][4], uint32_t st, uint32_t xs, int h, bool cvalid,
                                               int M, const uint32_t (&w_off)[kR][2], const uint32_t (&sf_off)[kR][2],
                                               uint32_t key, int g, int c) {
  const int j = 4 * h + c;
  uint4 A[kR][2];
  uint32_t slo[kR][2], shi[kR][2];
  const uint32_t sc_off = (j / 2) * 512 + 2 * (j % 2);
#pragma unroll
  for (int b = 0; b < kR; ++b) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      A[b][hr] = lds128(st + w_off[b][hr] + ((static_cast<uint32_t>(j) ^ key) * 16));
      scale_pair_to_bf16x2(lds16(st + sf_off[b][hr] + sc_off), slo[b][hr], shi[b][hr]);
      if (!cvalid) slo[b][hr] = shi[b][hr] = 0u;
    }
  }
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int kk = 32 * j + 8 * w;
    const uint32_t u = kk / 64, ch = (kk % 64) / 8;
    const uint4 xv =
        perm_x8(lds128_if(xs + (u * M + g) * 128 + ((ch ^ static_cast<uint32_t>(g)) * 16), g < M));
#pragma unroll
    for (int b = 0; b < kR; ++b) {
      const uint32_t w0 = w == 0 ? A[b][0].x : w == 1 ? A[b][0].y : w == 2 ? A[b][0].z : A[b][0].w;
      const uint32_t w1 = w == 0 ? A[b][1].x : w == 1 ? A[b][1].y : w == 2 ? A[b][1].z : A[b][1].w;
      uint32_t r0[4], r1[4];
      e2m1x8_raw_perm(w0, r0);
      e2m1x8_raw_perm(w1, r1);
      const uint32_t sa = w < 2 ? slo[b][0] : shi[b][0], sb = w < 2 ? slo[b][1] : shi[b][1];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        r0[q] = bf16x2_mul(r0[q], sa);
        r1[q] = bf16x2_mul(r1[q], sb);
      }
      mma_bf16_16816(accb[b], r0[0], r1[0], r0[1], r1[1], xv.x, xv.y);
      mma_bf16_16816(accb[b], r0[2], r1[2], r0[3], r1[3], xv.z, xv.w);
    }
  }
}

// kMode: kDenseFp4 (nvfp4_gemv); kMoeGateUp (the gate_up launch of
// vllm.models.flint.ops.moe_gemv: routed chunks of up to kSlabChunk pairs of
// one expert, and the shared expert's token chunks, with the epilogues of
// the register-fed kernel); kMoeDown (down_combine: chunks of up to 8 pairs;
// CTA column x streams its share of the row tiles (the tiles split evenly
// over gridDim.x groups) in turn over one resident activation slab, the
// whole K, and after each tile writes the
// tile's y rows, arrives on the tile's counter and, when it arrives last,
// combines the tile's outputs).
// kGroupedUp: gate_up in the grouped form (see below; down_combine always).
template <int kR, int kMode = kDenseFp4, bool kGroupedUp = false>
__global__ void __launch_bounds__(kSlabThreads, kSlabMinBlocks) gemv_slab_kernel(const __grid_constant__ GemvParams p) {
  using C = SlabCfg<kR>;
  constexpr int kChains = C::kChains;
  constexpr bool kDense = kMode == kDenseFp4;
  constexpr bool kDown = kMode == kMoeDown;
  static_assert(kDense || kMode == kMoeGateUp || kDown, "slab kernel modes");
  constexpr int kChunk = kDown ? kSlabNT : kSlabChunk;  // B rows of a MoE CTA, at most
  using Work = CtaWorkN<kChunk>;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t slab = base;                    // activations
  const uint32_t ring = base + p.x_off;          // weight stages (x_off: the slab's bytes, 1024-aligned)
  const uint32_t inbox = ring + p.nstages * p.stage_bytes;
  __shared__ __align__(8) uint64_t bar_full[kMaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t bar_inbox;
  __shared__ volatile int s_abort;
  // bit s: stage s has an activation that is not an exact f16 (down_combine:
  // every stage takes the shifted route)
  __shared__ uint32_t s_xbad[kSlabMaxStages / 32];
  // such a stage: largest / smallest biased exponent field of its nonzero
  // activations (its f16_shift); down_combine gathers them with atomics
  using ExpT = std::conditional_t<kDown, int, uint8_t>;
  __shared__ ExpT s_emax[kSlabMaxStages];
  __shared__ ExpT s_emin[kSlabMaxStages];
  __shared__ Work s_mwork;                // MoE: the CTA's work, resolved by the producer warp

  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;
  const int cw = p.cw;                 // consumer warps; warp cw is the producer
  const int ncons = cw * 32;
  const uint32_t S = cluster_nctarank();
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0;
  const int nstages = p.nstages;
  const int trows = 16 * kR * cw;

  // ---- what this CTA computes (dense: every thread derives it; MoE: the
  // producer warp resolves it -- routed CTAs after the router's ids are
  // complete -- and every thread copies it) ----
  RfWork wk;
  wk.shared = 0;
  wk.expert = -1;
  if constexpr (!kDense) {
    if (warp == cw) resolve_work<kMode, kChunk, Work>(p, s_mwork, 0, lane);
    __syncthreads();
    copy_work(s_mwork, wk);
    if constexpr (!kDown) {
      wk.k_begin = static_cast<int>(rank) * p.k_split;  // routed and shared K are both H
      wk.k_end = min(p.K, wk.k_begin + p.k_split);
    }
    // (down_combine: the whole K; the host sets routed_tiles = shared_tiles
    // = the tile groups, and the box is moved to the group's tiles below)
  } else {
    const int tile = blockIdx.x / max(1u, S);
    wk.k_begin = static_cast<int>(rank) * p.k_split;
    wk.k_end = min(p.K, wk.k_begin + p.k_split);
    wk.kbp = p.kbp;
    wk.sgroup[2] = wk.sgroup[3] = -1;
    wk.wrow[1] = wk.srow[1] = 0;
    const int groups_total = (p.rows_w + 127) / 128;
    if (p.silu) {
      wk.paired = 1;
      wk.out_base = tile * (trows / 2);
      rf_box(wk, 0, wk.out_base, trows / 2, groups_total);
      rf_box(wk, 1, p.n_half + wk.out_base, trows / 2, groups_total);
    } else {
      wk.paired = 0;
      wk.out_base = tile * trows;
      rf_box(wk, 0, wk.out_base, trows, groups_total);
    }
  }
  // B rows: tokens (dense) or the pairs of the expert chunk / the shared
  // expert's tokens (MoE; 0 for an inactive CTA, which streams nothing)
  const int M = kDense ? p.M : (s_mwork.active ? s_mwork.ntok : 0);
  const int klen = wk.k_end - wk.k_begin;
  const int nst_tile = (klen + 255) / 256;  // stages per row tile (and activation stages in the slab)
  // Tile groups (down_combine always; gate_up in the grouped form, with the
  // whole H per CTA): CTA column x takes the
  // tiles [x tiles / gridDim.x, (x + 1) tiles / gridDim.x) of its column's
  // weight in turn over one resident activation slab: 128-row tiles of H
  // (down_combine), [up; gate] groups of 64 features (routed gate_up) or
  // pairs of 64-row gate and up boxes (shared gate_up).
  constexpr bool grouped = kDown || (kMode == kMoeGateUp && kGroupedUp);
  const int tiles_h = kDown ? (p.n_out + 127) / 128
                            : (wk.shared ? (p.shared_n_out + 63) / 64 : p.n_out / 64);
  const int tile0 = grouped ? static_cast<int>(blockIdx.x * tiles_h / gridDim.x) : 0;
  const int ntl = grouped ? static_cast<int>((blockIdx.x + 1) * tiles_h / gridDim.x) - tile0 : 1;
  auto tile_of = [&](int tt) { return tile0 + tt; };  // tile index
  // The weight boxes of tile t (grouped modes).
  auto box_for_tile = [&](RfWork& w, int t) {
    if (kDown || !w.shared) {
      w.wrow[0] = (w.shared ? 0 : w.expert * p.rows_per_expert) + t * 128;
      w.srow[0] = t * 128;
      w.sgroup[0] = t;
    } else {
      const int groups_total = (p.rows_w + 127) / 128;
      rf_box(w, 0, t * 64, 64, groups_total);                 // gate rows
      rf_box(w, 1, p.n_half + t * 64, 64, groups_total);      // up rows
    }
  };
  if (grouped && ntl > 0) box_for_tile(wk, tile_of(0));
  const int nst = M > 0 && ntl > 0 ? ntl * nst_tile : 0;
  if (grouped && nst == 0) return;  // (uniform: no barrier, copy or arrival of this CTA is pending)
  const uint32_t slab_stage = static_cast<uint32_t>(M) * 512u;  // bytes of one stage's activations
  const uint64_t pol_w = policy_evict_first();
  auto issue_weights = [&](int s, int slot) {
    const uint32_t st = ring + slot * p.stage_bytes;
    const uint32_t fb = smem_u32(&bar_full[slot]);
    int tt = 0, ks = s;  // row tile (grouped modes) and K stage
    RfWork bw = wk;
    if constexpr (grouped) {
      tt = s / nst_tile;
      ks = s - tt * nst_tile;
      box_for_tile(bw, tile_of(tt));
    }
    const int k0 = wk.k_begin + ks * 256;
    const int nchunks = min(256, wk.k_end - k0) / kSubK;
    const CUtensorMap* tmw = wk.shared ? &p.tm_w2 : &p.tm_w;
    const uint8_t* sfb =
        wk.shared ? p.sf2 : p.sf + (wk.expert >= 0 ? static_cast<size_t>(wk.expert) * p.sf_expert_bytes : 0);
    uint32_t bytes = trows * 128;
#pragma unroll
    for (int g = 0; g < 4; ++g) bytes += (bw.sgroup[g] >= 0 ? nchunks * 512 : 0);
    mbar_arrive_expect_tx(fb, bytes);
    tma_load_2d(st, tmw, k0 / 2, bw.wrow[0], fb, pol_w);
    if (bw.paired) tma_load_2d(st + trows * 64, tmw, k0 / 2, bw.wrow[1], fb, pol_w);
    uint32_t sdst = st + trows * 128;  // the valid groups, in order
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (bw.sgroup[g] < 0) continue;
      const size_t chunk = static_cast<size_t>(bw.sgroup[g]) * (wk.kbp / 4) + k0 / 64;
      bulk_load(sdst, sfb + chunk * 512, nchunks * 512, fb, pol_w);
      sdst += 2048;
    }
  };
  // Output rows are reduced across cluster ranks per feature unit: paired
  // tiles and routed [up; gate] groups combine rows o and o + trows / 2 (two
  // rows per feature).
  const int unit = (wk.paired || !kDense) ? trows / 2 : trows;
  const int rpf = trows / unit;

  // ------------------------------------------------------------------ prologue
  if (warp == cw && lane == 0) {
    prefetch_tensormap(&p.tm_w);
    if constexpr (!kDense) prefetch_tensormap(&p.tm_w2);
    s_abort = 0;
    for (int i = 0; i < nstages; ++i) {
      mbar_init(smem_u32(&bar_full[i]), 1);
      mbar_init(smem_u32(&bar_empty[i]), cw);
    }
    mbar_init(smem_u32(&bar_inbox), 1);
    if (S > 1) {
      const int r = (unit + static_cast<int>(S) - 1) / static_cast<int>(S);
      const int mine0 = max(0, min(r, unit - static_cast<int>(rank) * r)) * rpf;
      mbar_arrive_expect_tx(smem_u32(&bar_inbox), S * M * mine0 * 4);  // tokens < M only
    }
    mbar_fence_init();
    const int pre = min(nst, nstages);
    for (int s = 0; s < pre; ++s)
      if (s != p.skip_stage) issue_weights(s, s);  // (test hook: the skipped stage is never issued)
  }
  for (int i = tid; i < kSlabMaxStages / 32; i += blockDim.x) s_xbad[i] = kDown ? 0xFFFFFFFFu : 0u;
  if constexpr (kDown) {
    for (int i = tid; i < nst_tile; i += blockDim.x) {
      s_emax[i] = 0;
      s_emin[i] = 255;
    }
  }
  __syncthreads();
  if (S > 1) cluster_arrive_relaxed();  // paired with a wait before the first remote access
  if (tid == 0) pdl_launch_dependents();
  const int R = (unit + static_cast<int>(S) - 1) / static_cast<int>(S);
  const int f_lo = static_cast<int>(rank) * R;
  const int f_hi = min(unit, f_lo + R);
  const int mine = max(0, f_hi - f_lo) * rpf;

  float acc[kChains][kR][4];   // f16-route stages (exact products)
  float accb[kR][4];           // bf16-route stages (products times 2^-kShift)
#pragma unroll
  for (int b = 0; b < kR; ++b) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      accb[b][e] = 0.0f;
#pragma unroll
      for (int q = 0; q < kChains; ++q) acc[q][b][e] = 0.0f;
    }
  }
  const int g = lane / 4, c = lane % 4;
  const int sg = (g % 2) * 4 + g / 2;  // sigma(g)
  // Tile row of this thread's MMA row sg + 8 hr in row block b.  gate_up's
  // grouped form pairs a feature's two rows in one thread: warp w's block 0
  // holds rows 16 w .. 16 w + 15 and block 1 the rows 64 below them (a
  // routed [up; gate] group's up and gate rows, a shared pair's gate and up
  // rows), so the tile epilogue needs no exchange.  Other forms: the warp's
  // kR consecutive 16-row blocks.
  constexpr bool kPairRows = kMode == kMoeGateUp && kGroupedUp;
  static_assert(!kPairRows || kR == 2, "paired rows: two 16-row blocks per warp, 128-row tiles");
  auto tile_row = [&](int b, int hr) {
    return kPairRows ? b * 64 + warp * 16 + sg + 8 * hr : (warp * kR + b) * 16 + sg + 8 * hr;
  };

  if (warp == cw) {
    // ------------------------------------------------------------------ producer
    // Weights only; they do not depend on the previous grid, so no wait.
    if (lane == 0) {
      const int pre = min(nst, nstages);
      int issued = pre;
      for (int s = pre, slot = pre % nstages, ph = (pre / nstages) & 1; s < nst && !s_abort;
           ++s, slot = slot + 1 == nstages ? 0 : slot + 1, ph ^= slot == 0) {
        if (!mbar_wait_sleepy(smem_u32(&bar_empty[slot]), ph ^ 1, p.err, 64)) {
          s_abort = 1;
          break;
        }
        if (s != p.skip_stage) issue_weights(s, slot);
        issued = s + 1;
      }
      // After an abort, let every copy still in flight land before the CTA
      // (and its shared memory) goes away: the latest fill of each slot.
      if (s_abort) {
        for (int s = max(0, issued - nstages); s < issued; ++s)
          if (s != p.skip_stage) (void)mbar_wait(smem_u32(&bar_full[s % nstages]), (s / nstages) & 1, p.err);
      }
    }
  } else {
    // ------------------------------------------------------------------ consumers
    // The activation slab: bf16 chunks in (pass 1, with an exactness check
    // per stage); stages with an inexact value get their exponent range (pass
    // 1b, only if there are any); then the exact stages to f16 in place and
    // the others with an f16 shift to x 2^s (pass 2); the rest stay bf16 for
    // the bf16 route.  down_combine, whose activations (gate_up's outputs)
    // are often not all exact f16s, takes every stage's range in pass 1 and
    // shifts every stage (a measured 4 % on the call).
    // K past the end of a ragged last stage is zero-filled (the same bits in
    // bf16 and f16), so the zero weights there meet zero activations.
    pdl_wait();
    const int nchk = klen / 8;  // 16-byte chunks per token holding data
    const int nslot = (M > 0 ? nst_tile : 0) * 32;  // 16-byte chunks per token in the slab
    // (loads in batches of kFillBatch per thread, all issued before their
    // stores, so a thread waits for one round trip per batch, not per chunk)
    constexpr int kFillBatch = 4;
    for (int q0 = tid; q0 < M * nslot; q0 += kFillBatch * ncons) {
      uint4 v[kFillBatch];
#pragma unroll
      for (int i = 0; i < kFillBatch; ++i) {
        const int q = q0 + i * ncons;
        const int n = q / nslot, kq = q % nslot;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (q < M * nslot && kq < nchk) {
          const uint16_t* xr = kDense ? p.x + static_cast<int64_t>(n) * p.ldx
                                      : (wk.shared ? p.x2 : p.x) + s_mwork.xoff[n];
          v[i] = __ldg(reinterpret_cast<const uint4*>(xr + wk.k_begin + 8 * kq));
        }
      }
#pragma unroll
      for (int i = 0; i < kFillBatch; ++i) {
        const int q = q0 + i * ncons;
        if (q >= M * nslot) break;
        const int n = q / nslot, kq = q % nslot;
        const int s = kq / 32, u = (kq % 32) / 8, ch = kq % 8;
        const uint32_t a = slab + s * slab_stage + (u * M + n) * 128 + ((ch ^ (n & 7)) * 16);
        sts128(a, v[i]);
        if constexpr (kDown) {
          // (a warp's 32 chunks share a token and a stage: M nslot and nslot
          // are multiples of 32, and so is the first q of every warp)
          int emx, emn;
          bf16x8_exp_range(v[i], emx, emn);
          emx = __reduce_max_sync(0xFFFFFFFFu, emx);
          emn = __reduce_min_sync(0xFFFFFFFFu, emn);
          if (lane == 0) {
            atomicMax(&s_emax[s], emx);
            atomicMin(&s_emin[s], emn);
          }
        } else {
          uint4 o;
          if (!bf16x8_to_f16x8_exact(v[i], o)) atomicOr(&s_xbad[s / 32], 1u << (s % 32));
        }
      }
    }
    cons_sync(ncons);
    auto xbad = [&](int s) { return (s_xbad[s / 32] >> (s % 32)) & 1u; };
    bool any_bad = false;
    for (int i = 0; i < kSlabMaxStages / 32; ++i) any_bad |= s_xbad[i] != 0u;
    if (!kDown && any_bad) {
      // one warp per such stage: the exponent range of its M x 32 chunks
      // (chunks past the end of K hold zeros)
      for (int s = warp; s < nst_tile; s += cw) {
        if (!xbad(s)) continue;
        int emx = 0, emn = 255;
        for (int q = lane; q < M * 32; q += 32) {
          const int n = q / 32, u = (q % 32) / 8, ch = q % 8;
          int e1, e2;
          bf16x8_exp_range(lds128(slab + s * slab_stage + (u * M + n) * 128 + ((ch ^ (n & 7)) * 16)), e1, e2);
          emx = max(emx, e1);
          emn = min(emn, e2);
        }
        emx = __reduce_max_sync(0xFFFFFFFFu, emx);
        emn = __reduce_min_sync(0xFFFFFFFFu, emn);
        if (lane == 0) {
          s_emax[s] = static_cast<uint8_t>(emx);
          s_emin[s] = static_cast<uint8_t>(emn);
        }
      }
      cons_sync(ncons);
    }
    for (int q = tid; q < M * nchk; q += ncons) {
      const int n = q / nchk, kq = q % nchk;
      const int s = kq / 32, u = (kq % 32) / 8, ch = kq % 8;
      const uint32_t a = slab + s * slab_stage + (u * M + n) * 128 + ((ch ^ (n & 7)) * 16);
      if (!kDown && !xbad(s)) {
        uint4 o;
        bf16x8_to_f16x8_exact(lds128(a), o);
        sts128(a, o);
        continue;
      }
      const int sh = f16_shift(s_emax[s], s_emin[s]);
      if (sh >= 0) sts128(a, bf16x8_to_f16x8_scaled(lds128(a), __int_as_float((127 + sh) << 23)));
    }
    cons_sync(ncons);

    // shared-memory offsets of this thread's rows (128-byte swizzle key
    // = row % 8, the same for every row of the thread) and of their scales
    uint32_t w_off[kR][2], sf_off[kR][2];
    const uint32_t key = static_cast<uint32_t>(sg);
    auto set_offsets = [&](const RfWork& w) {
#pragma unroll
      for (int b = 0; b < kR; ++b) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int row = tile_row(b, hr);
          w_off[b][hr] = (row / 8) * 1024 + (row % 8) * 128;
          const int half = trows / 2;
          const bool b1 = w.paired && row >= half;
          const int r = (b1 ? w.srow[1] : w.srow[0]) + (b1 ? row - half : row);
          const int gr = r / 128;
          const int gslot = b1 ? (w.sgroup[0] >= 0) + (w.sgroup[1] >= 0) + (gr != w.sgroup[2]) : (gr != w.sgroup[0]);
          sf_off[b][hr] = trows * 128 + gslot * 2048 + (r % 32) * 16 + ((r % 128) / 32) * 4;
        }
      }
    };
    set_offsets(wk);
    // After a tile's last stage (grouped modes).  Every consumer warp calls
    // it for the same tiles, also after a wait ran out; returns the abort.
    // The accumulators restart.
    //   down_combine: the tile's y rows (y_j = bf16(acc * alpha2[e]) into
    //     the workspace, or y_shared = bf16(acc * gssd)), each warp its own
    //     rows with no barrier: the combine is a kernel of its own, after
    //     this grid.  A CTA that gave up tags its tiles instead (below).
    //   gate_up (grouped form): each thread holds both rows of its features
    //     (tile_row) and writes their outputs, with no barrier; a warp that
    //     saw a wait run out writes nothing (the tile's outputs stay
    //     unwritten).  Otherwise the tile's sums are staged in shared memory
    //     (row-major per B row), then the 64 features' outputs as in the
    //     split epilogue; the first barrier agrees on the abort.
    auto tile_done = [&](int tt) -> bool {
      const bool ab = (kDown || kPairRows) ? s_abort != 0 : bar_red_or<1>(ncons, s_abort != 0);
      const int t = tile_of(tt);
      const float post = static_cast<float>(1 << kShift);
      float v[kR][2][2];  // this thread's sums: row block, row half, token
#pragma unroll
      for (int b = 0; b < kR; ++b) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float a = accb[b][2 * hr + e] * post;
            accb[b][2 * hr + e] = 0.0f;
#pragma unroll
            for (int q = 0; q < kChains; ++q) {
              a += acc[q][b][2 * hr + e];
              acc[q][b][2 * hr + e] = 0.0f;
            }
            v[b][hr][e] = a;
          }
        }
      }
      if constexpr (kDown) {
        const int h0 = t * 128;
        if (!ab) {
          const float sc = wk.shared ? __ldg(p.gs) : __ldg(p.alpha + wk.expert);
          uint16_t* dst = wk.shared ? p.out2 : p.out;
          const int64_t ld = wk.shared ? p.ldo2 : p.ldo;
#pragma unroll
          for (int b = 0; b < kR; ++b) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              const int h = h0 + (warp * kR + b) * 16 + sg + 8 * hr;
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int n = 2 * c + e;
                if (n < M && h < p.n_out)
                  dst[static_cast<int64_t>(s_mwork.orow[n]) * ld + h] = f32_to_bf16_rn(v[b][hr][e] * sc);
              }
            }
          }
        }
      } else if constexpr (kPairRows) {
        // this thread's features 16 w + sg + 8 hr, tokens 2 c + e: block 0
        // holds the up (routed) or gate (shared) row, block 1 the other
        if (!ab) {
          const float sc = wk.shared ? __ldg(p.gs) : __ldg(p.alpha + wk.expert);
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int feat = t * 64 + warp * 16 + sg + 8 * hr;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int n = 2 * c + e;
              if (n >= M) continue;
              if (!wk.shared) {
                if (feat < p.n_out)
                  p.out[static_cast<int64_t>(s_mwork.orow[n]) * p.ldo + feat] =
                      f32_to_bf16_rn(silu_fast(v[1][hr][e] * sc) * (v[0][hr][e] * sc));
              } else if (feat < p.shared_n_out) {
                const float G = bf16_to_f32(f32_to_bf16_rn(v[0][hr][e] * sc));
                const float U = bf16_to_f32(f32_to_bf16_rn(v[1][hr][e] * sc));
                p.out2[static_cast<int64_t>(s_mwork.orow[n]) * p.ldo2 + feat] = f32_to_bf16_rn(silu_exact(G) * U);
              }
            }
          }
        }
      } else {
        if (!ab) {
#pragma unroll
          for (int b = 0; b < kR; ++b) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              const int row = tile_row(b, hr);
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int n = 2 * c + e;
                if (n < M) stsf(inbox + (n * 128 + row) * 4, v[b][hr][e]);
              }
            }
          }
        }
        cons_sync(ncons);
        if (!ab) {
          if (!wk.shared) {
            // routed [up; gate] group: feature o = up row o, gate row o + 64
            const float al = __ldg(p.alpha + wk.expert);
            for (int it = tid; it < 64 * M; it += ncons) {
              const int n = it / 64, lr = it % 64;
              const int feat = t * 64 + lr;
              if (feat >= p.n_out) continue;
              const float uu = ldsf(inbox + (n * 128 + lr) * 4) * al;
              const float gt = ldsf(inbox + (n * 128 + 64 + lr) * 4) * al;
              p.out[static_cast<int64_t>(s_mwork.orow[n]) * p.ldo + feat] = f32_to_bf16_rn(silu_fast(gt) * uu);
            }
          } else {
            // shared expert: feature o = gate row o, up row o + 64
            const float gs = __ldg(p.gs);
            for (int it = tid; it < 64 * M; it += ncons) {
              const int n = it / 64, lr = it % 64;
              const int feat = t * 64 + lr;
              if (feat >= p.shared_n_out) continue;
              const float G = bf16_to_f32(f32_to_bf16_rn(ldsf(inbox + (n * 128 + lr) * 4) * gs));
              const float U = bf16_to_f32(f32_to_bf16_rn(ldsf(inbox + (n * 128 + 64 + lr) * 4) * gs));
              p.out2[static_cast<int64_t>(s_mwork.orow[n]) * p.ldo2 + feat] = f32_to_bf16_rn(silu_exact(G) * U);
            }
          }
        }
      }
      return ab;
    };
    for (int s = 0, slot = 0, ph = 0; s < nst; ++s, slot = slot + 1 == nstages ? 0 : slot + 1, ph ^= slot == 0) {
      const uint32_t st = ring + slot * p.stage_bytes;
      const int tt = grouped ? s / nst_tile : 0;  // tile (grouped modes)
      const int ks = s - tt * nst_tile;           // K stage
      const uint32_t xs = slab + ks * slab_stage;
      if (grouped && ks == 0 && tt > 0) {
        // (the scale offsets of shared gate_up boxes move with the tile)
        RfWork tw = wk;
        box_for_tile(tw, tile_of(tt));
        set_offsets(tw);
      }
      const bool ok = __all_sync(0xFFFFFFFFu, !s_abort && mbar_wait(smem_u32(&bar_full[slot]), ph, p.err));
      if (!ok) {
        s_abort = 1;
        if constexpr (grouped) {
          // (the slot is not released: its copy may still land)
          if (ks == nst_tile - 1 && tile_done(tt)) break;
          continue;
        }
        break;
      }
      // valid K of the stage: 64 .. 256 in steps of 64; a chunk (32 K) is
      // wholly valid or wholly past the end
      const int kvalid = min(256, klen - ks * 256);
      const bool bad = kDown || ((s_xbad[ks / 32] >> (ks % 32)) & 1u);
      const int sh = bad ? f16_shift(s_emax[ks], s_emin[ks]) : 0;
      if (!bad) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (128 * h < kvalid) {
            if (128 * (h + 1) <= kvalid)
              slab_half_f16<kR, kChains, false>(acc, st, xs, h, true, M, w_off, sf_off, key, g, c, 0u);
            else
              slab_half_f16<kR, kChains, false>(acc, st, xs, h, 32 * (4 * h + c) < kvalid, M, w_off, sf_off, key, g, c, 0u);
          }
        }
      } else if (sh >= 0) {
        const uint32_t sdown = f16x2_pow2_neg(sh);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (128 * h < kvalid) {
            if (128 * (h + 1) <= kvalid)
              slab_half_f16<kR, kChains, true>(acc, st, xs, h, true, M, w_off, sf_off, key, g, c, sdown);
            else
              slab_half_f16<kR, kChains, true>(acc, st, xs, h, 32 * (4 * h + c) < kvalid, M, w_off, sf_off, key, g, c, sdown);
          }
        }
      } else {
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          if (128 * h < kvalid) slab_half_bf16<kR>(accb, st, xs, h, 32 * (4 * h + c) < kvalid, M, w_off, sf_off, key, g, c);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_empty[slot]));
      if (grouped && ks == nst_tile - 1 && tile_done(tt)) break;
    }
  }

  // ==================================================================== epilogue
  __syncwarp();
  if constexpr (grouped) {
    // (grouped modes finished each tile inside the loop)
  } else if (warp < cw) {
    const float post = static_cast<float>(1 << kShift);
    // Push this thread's partials (its rows, tokens 2c + {0,1} below M) to
    // the owners of the rows: inbox[src][n][rr].
    if (S > 1) cluster_wait();  // all peers' inbox barriers are initialised
    const bool go = !s_abort;
#pragma unroll
    for (int b = 0; b < kR; ++b) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = (warp * kR + b) * 16 + sg + 8 * hr;
        const int fi = row % unit;
        const int owner = fi / R;
        const int owner_feats = min(R, unit - owner * R);
        const int rr = (row / unit) * owner_feats + (fi - owner * R);
        const int rows_owner = owner_feats * rpf;
        const uint32_t bse = inbox + ((rank * M) * rows_owner + rr) * 4;
        const uint32_t rbase = S > 1 ? mapa(bse, static_cast<uint32_t>(owner)) : bse;
        const uint32_t rbar = S > 1 ? mapa(smem_u32(&bar_inbox), static_cast<uint32_t>(owner)) : 0u;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int n = 2 * c + e;
          float a16 = 0.0f;
#pragma unroll
          for (int q = 0; q < kChains; ++q) a16 += acc[q][b][2 * hr + e];
          a16 += accb[b][2 * hr + e] * post;
          const float v = go ? a16 : 0.0f;
          if (n >= M) continue;
          const uint32_t off = n * rows_owner * 4;
          if (S > 1) st_async_f32(rbase + off, v, rbar);
          else stsf(rbase + off, v);
        }
      }
    }
    if (S > 1) {
      if (!mbar_wait<true>(smem_u32(&bar_inbox), 0, p.err)) s_abort = 1;
    } else {
      cons_sync(ncons);
    }
    auto partial = [&](int n, int lr) -> float {
      float a = 0.0f;
      for (uint32_t src = 0; src < S; ++src) a += ldsf(inbox + ((src * M + n) * mine + lr) * 4);
      return a;
    };
    const int nf = f_hi - f_lo;
    if (!s_abort && nf > 0 && !kDense) {
      if (!wk.shared) {
        // routed [up; gate] group: feature o = up row o, gate row o + 64
        const float al = __ldg(p.alpha + wk.expert);
        for (int it = tid; it < nf * M; it += ncons) {
          const int n = it / nf, lr = it % nf;
          const int feat = wk.out_base + f_lo + lr;
          if (feat >= p.n_out) continue;
          const float uu = partial(n, lr) * al;
          const float gt = partial(n, lr + nf) * al;
          p.out[static_cast<int64_t>(s_mwork.orow[n]) * p.ldo + feat] = f32_to_bf16_rn(silu_fast(gt) * uu);
        }
      } else {
        // shared expert, paired tiles: feature o = gate row o, up row o + 64
        const float gs = __ldg(p.gs);
        for (int it = tid; it < nf * M; it += ncons) {
          const int n = it / nf, lr = it % nf;
          const int feat = wk.out_base + f_lo + lr;
          if (feat >= p.shared_n_out) continue;
          const float G = bf16_to_f32(f32_to_bf16_rn(partial(n, lr) * gs));
          const float U = bf16_to_f32(f32_to_bf16_rn(partial(n, lr + nf) * gs));
          p.out2[static_cast<int64_t>(s_mwork.orow[n]) * p.ldo2 + feat] = f32_to_bf16_rn(silu_exact(G) * U);
        }
      }
    } else if (!s_abort && nf > 0) {
      const float gs = __ldg(p.gs);
      if (rpf == 1) {
        for (int it = tid; it < nf * M; it += ncons) {
          const int n = it / nf, lr = it % nf;
          const int o = wk.out_base + f_lo + lr;
          if (o >= p.n_out) continue;
          p.out[static_cast<int64_t>(n) * p.ldo + o] = f32_to_bf16_rn(partial(n, lr) * gs);
        }
      } else {
        // paired tiles: feature o = gate row o, up row o + unit
        for (int it = tid; it < nf * M; it += ncons) {
          const int n = it / nf, lr = it % nf;
          const int feat = wk.out_base + f_lo + lr;
          if (feat >= p.n_out) continue;
          const float G = bf16_to_f32(f32_to_bf16_rn(partial(n, lr) * gs));
          const float U = bf16_to_f32(f32_to_bf16_rn(partial(n, lr + nf) * gs));
          p.out[static_cast<int64_t>(n) * p.ldo + feat] = f32_to_bf16_rn(silu_exact(G) * U);
        }
      }
    }
  } else if (S > 1) {
    cluster_wait();  // the producer warp closes its cluster-barrier phase
  }
  __syncthreads();
  // down_combine: a CTA that gave up tags each of its tiles with this call's
  // epoch, and the combine kernel leaves those tiles' outputs unwritten.
  if (kDown && tid == 0 && s_abort)
    for (int tt = 0; tt < ntl; ++tt) p.counters[tile_of(tt)] = abort_tag(p.epoch);
}

}  // namespace fp4
