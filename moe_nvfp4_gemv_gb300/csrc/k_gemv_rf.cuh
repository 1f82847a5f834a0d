// k_gemv_rf.cuh -- the NVFP4 GEMV for M <= 16 with register-fed MMAs: the
// dense calls the slab kernel (k_gemv_slab.cuh) does not serve, and the MoE
// calls of up to 64 tokens (chunks of up to 8 pairs) it has no plan for.
//
// Same operation as the dense mode of k_gemv.cuh (vllm.models.flint.ops.nvfp4_gemv
// nvfp4_gemv, with or without silu_mul), built for the decode shapes where
// the token count is tiny.  On this GPU a tcgen05 MMA with N <= 64 costs about
// as much as N = 64 (a 128x16x16 MMA occupies the tensor core ~46 cycles,
// plus ~44 per commit), which caps a swap-AB tcgen05 GEMV near the HBM rate
// with no headroom.  The warp-level m16n8k16 MMA processes a 16-row x 16-K
// weight block for 8 tokens at ~0.4 per cycle per SM (~100 weights per cycle
// per SM), so it is not the bottleneck; the dequantization is.
//
// Layout of the work: a CTA owns one weight tile of 16 cw rows (plain, or 8 cw
// gate + 8 cw up rows for silu_mul; cw = 6..8 consumer warps for the dense
// GEMV, chosen per call, 8 for MoE) and a K range; the S CTAs of a cluster
// split K and reduce in rank order through distributed shared memory, as the
// tcgen05 kernel does.  A producer warp streams weights, scales and
// activations into a ring of 256-K stages (TMA / bulk copies, weights issued
// before griddepcontrol.wait).  Each working consumer warp owns 16 rows of
// the tile; per stage it reads its rows' codes and scales from shared memory,
// dequantizes them exactly in registers (dequant.cuh) straight into MMA A
// fragments, loads the activation B fragments and accumulates in fp32
// registers.  Warps meet only through the stage ring (and, in the
// cooperative variant, at one barrier per stage).
//
// Fragment mapping.  Thread (g, c) = (lane / 4, lane % 4) of warp wp holds
// MMA rows g and g + 8, which are tile rows 16 wp + sigma(g) and
// 16 wp + 8 + sigma(g), sigma = (0 4 1 5 2 6 3 7): neighbouring g then sit in
// different halves of the 128-byte swizzle, so the 16-byte code loads of a
// quarter warp hit distinct banks.  In each 128-K half h of a stage thread c
// reads code chunk j = 4 h + c (32 codes) of both rows; word w of the chunk
// (8 codes) yields the bf16 pairs (c0,c4) (c2,c6) (c1,c5) (c3,c7), the A
// registers of two MMAs, and the activation chunk of the same 8 K (token g,
// permuted the same way) their B registers.
//
// Routes.  The bf16 route above serves 13-16 tokens (and MoE chunks of 5-8
// pairs).  For M <= kF16MaxM the f16 route: a converter warp turns each
// stage's activation rows in shared memory into f16 in place as soon as they
// land (ahead of the consumers: its arrival is part of the stage's full
// barrier, so a consumer waits on one barrier per stage), checking that every
// value converts exactly; the stage then runs on f16 MMAs with the codes
// converted by cvt.rn.f16x2.e2m1x2 (natural K order, half the ALU work of the
// bf16 route).  The dense variant for 3-12 tokens (kCoop, 8- and 16-token
// tiles) converts with all consumer warps instead.  A stage with any value that is not exactly an f16 (|x| > 65504,
// too many low bits for the f16 subnormal grid, NaN) runs the bf16 route with
// the original activations from global memory instead.  Both routes compute
// exact products into fp32, so the choice changes no result beyond fp32
// accumulation order; they accumulate separately (the bf16 route's products
// carry the 2^-kShift factor) and are summed at the end.
#pragma once

#include "k_gemv.cuh"

namespace fp4 {

template <int kNT>
struct RfCfg {
  static constexpr int kConsumerWarps = 8;
  static constexpr int kThreads = kConsumerWarps * 32 + 64;
  static constexpr int kProducerWarp = kConsumerWarps;
  static constexpr int kConverterWarp = kConsumerWarps + 1;
  static constexpr int kStageK = 256;
  // A stage: the weight tile (16 cw rows x 128 bytes), then 2 KB per 128-row
  // scale group its boxes touch (up to 4), then the activations; the host sets
  // the geometry per call (stage_bytes, x_off) so the ring is as deep as
  // shared memory allows.
  static constexpr int kXBytes = kNT * kStageK * 2;
  static constexpr int kTiles = kNT / 8;  // MMA n-tiles
  // Independent fp32 accumulators per n-tile on the f16 route: consecutive
  // MMAs of a thread go to different chains so they do not wait on each
  // other's results (an MMA's latency is several times its issue interval).
  static constexpr int kChains = kNT == 8 ? 4 : 1;  // (16 tokens: the two n-tiles already alternate)
  // Token counts up to which the f16 route is used: its per-stage activation
  // conversion (one warp) costs ~M x 32 chunk conversions, which outweighs
  // the cheaper dequantization beyond a few tokens.
  static constexpr int kF16MaxM = 4;
  static constexpr bool kHasF16 = kNT == 8;  // only the 8-token tile serves M <= kF16MaxM
  // The split-K inbox, then (MoE modes) the CTA's resolved work.
  static constexpr int kInboxFloats = kNT * 136;
  static constexpr int kWorkBytes = static_cast<int>((sizeof(CtaWork) + 15) / 16 * 16);
  static_assert(kNT == 8 || kNT == 16, "token tile");
};

// D += A * B for one m16n8k16 f16 MMA (fp32 accumulate).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte shared load that only lanes with `on` perform; the others get zeros
// (a predicated load: no branch, no shared-memory traffic for them).
__device__ __forceinline__ uint4 lds128_if(uint32_t a, bool on) {
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  asm volatile(
      "{ .reg .pred p; setp.ne.u32 p, %5, 0; @p ld.shared.v4.u32 {%0, %1, %2, %3}, [%4]; }"
      : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
      : "r"(a), "r"(static_cast<uint32_t>(on)));
  return v;
}

// Named barrier `id` over `count` threads that returns whether any of them
// passed `pred` true (also orders their shared-memory accesses).
template <int id>
__device__ __forceinline__ bool bar_red_or(uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

// D += A * B for one m16n8k16 bf16 MMA (fp32 accumulate).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The per-thread copy of a CTA's work: K range and the weight boxes
// (tensor-map rows, scale rows and groups).  Box b's rows lie in the 128-row
// scale groups sgroup[2b] and (when it straddles a boundary) sgroup[2b + 1];
// -1 marks none.  A stage holds the valid groups in this order, 2 KB each.
struct RfWork {
  int paired, shared, expert, k_begin, k_end, kbp, out_base;
  int wrow[2], srow[2], sgroup[4];
};

// Box b: weight rows [row, row + h), whose scales start at scale row `row`.
__device__ __forceinline__ void rf_box(RfWork& w, int b, int row, int h, int groups_total) {
  w.wrow[b] = row;
  w.srow[b] = row;
  const int g0 = row / 128, g1 = (row + h - 1) / 128;
  w.sgroup[2 * b] = g0 < groups_total ? g0 : -1;
  w.sgroup[2 * b + 1] = (g1 != g0 && g1 < groups_total) ? g1 : -1;
}

template <typename Work>
__device__ __forceinline__ void copy_work(const Work& m, RfWork& w) {
  w.paired = m.paired;
  w.shared = m.shared;
  w.expert = m.expert;
  w.k_begin = m.k_begin;
  w.k_end = m.k_end;
  w.kbp = m.kbp;
  w.out_base = m.out_base;
  w.wrow[0] = m.wrow[0];
  w.wrow[1] = m.wrow[1];
  w.srow[0] = m.srow[0];
  w.srow[1] = m.srow[1];
  w.sgroup[0] = m.sgroup[0];  // a 128-row box on a 128-row boundary: one group
  w.sgroup[1] = -1;
  w.sgroup[2] = m.sgroup[1];
  w.sgroup[3] = m.sgroup[2];
}

// kMode: kDenseFp4 (nvfp4_gemv), kMoeGateUp or kMoeDown (the same modes and
// epilogues as the tcgen05 kernel, for chunks of at most 16 tokens / pairs).
// kOcc: CTAs per SM the registers are budgeted for.  2 by default; 3 (two
// accumulator chains, 64 registers, the host gives it a 72 KB ring) for
// grids of many short CTAs, whose fixed costs more co-resident CTAs hide.
// kCoop: the dense variant for 3 .. 12 tokens whose consumer warps convert
// the activations to f16 together (a separate instantiation, so the others'
// code is unchanged by it).
template <int kMode, int kNT, int kOcc = 2, bool kCoop = false>
__global__ void __launch_bounds__(RfCfg<kNT>::kThreads, kOcc) gemv_rf_kernel(const __grid_constant__ GemvParams p) {
  using C = RfCfg<kNT>;
  constexpr int kChains = kOcc >= 3 && C::kChains > 2 ? 2 : C::kChains;
  // f16-route code: the 8-token tile (converter warp or cooperative) and the
  // cooperative variants of larger tiles
  constexpr bool kF16 = C::kHasF16 || kCoop;
  constexpr bool kDense = kMode == kDenseFp4;
  constexpr int kEpiThreads = C::kConsumerWarps * 32;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t inbox = ring + p.nstages * p.stage_bytes;
  __shared__ __align__(8) uint64_t bar_full[kMaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kMaxStages];
  // f16 route: the activations land on bar_xfull; the converter waits there and
  // its arrival (after the conversion) is one of the two that complete bar_full,
  // so the consumers wait on a single barrier per stage.
  __shared__ __align__(8) uint64_t bar_xfull[kMaxStages];
  __shared__ __align__(8) uint64_t bar_inbox;
  __shared__ volatile int s_abort;
  __shared__ int s_xbad[kMaxStages];  // last stage (of this slot) whose activations are not all exact f16
  __shared__ int s_last;
  // MoE: the CTA's work, resolved by the producer before the weight stream starts
  CtaWork* const mwork = reinterpret_cast<CtaWork*>(smem_raw + (inbox - smem_u32(smem_raw)) + C::kInboxFloats * 4);

  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;
  const uint32_t S = cluster_nctarank();
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0;
  const int nstages = p.nstages;

  // Dense tiles are 16 cw rows (cw consumer warps, chosen per call so the
  // grid fills the GPU evenly): 16 cw features, or with silu_mul 8 cw gate
  // rows and the 8 cw matching up rows.  MoE tiles are 128 rows.
  const int cw = kDense ? p.cw : C::kConsumerWarps;
  const int trows = 16 * cw;

  // ---- what this CTA computes (dense: every thread derives it) ----
  RfWork wk;
  wk.shared = 0;
  wk.expert = -1;
  if constexpr (kDense) {
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
  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_x = policy_evict_last();
  auto issue_weights = [&](int s, int slot) {
    const uint32_t st = ring + slot * p.stage_bytes;
    const uint32_t fb = smem_u32(&bar_full[slot]);
    const int k0 = wk.k_begin + s * C::kStageK;
    const int nchunks = min(C::kStageK, wk.k_end - k0) / kSubK;
    const CUtensorMap* tmw = wk.shared ? &p.tm_w2 : &p.tm_w;
    const uint8_t* sfb =
        wk.shared ? p.sf2 : p.sf + (wk.expert >= 0 ? static_cast<size_t>(wk.expert) * p.sf_expert_bytes : 0);
    uint32_t bytes = trows * 128;
#pragma unroll
    for (int g = 0; g < 4; ++g) bytes += (wk.sgroup[g] >= 0 ? nchunks * 512 : 0);
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(fb), "r"(bytes) : "memory");
    tma_load_2d(st, tmw, k0 / 2, wk.wrow[0], fb, pol_w);
    if (wk.paired) tma_load_2d(st + trows * 64, tmw, k0 / 2, wk.wrow[1], fb, pol_w);
    uint32_t sdst = st + trows * 128;  // the valid groups, in order
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (wk.sgroup[g] < 0) continue;
      const size_t chunk = static_cast<size_t>(wk.sgroup[g]) * (wk.kbp / 4) + k0 / 64;
      bulk_load(sdst, sfb + chunk * 512, nchunks * 512, fb, pol_w);
      sdst += 2048;
    }
  };
  // Output rows are reduced across cluster ranks per feature unit: a tile
  // whose feature o combines rows o and o + unit (paired gate/up boxes, routed
  // [up; gate] groups) has half-tile units and two rows per feature, any other
  // tile one row per feature.
  auto unit_of = [&]() {
    if constexpr (kDense) return wk.paired ? trows / 2 : trows;
    else return (wk.paired || (kMode == kMoeGateUp && !wk.shared)) ? 64 : 128;
  };
  auto rpf_of = [&]() { return trows / unit_of(); };
  auto stages_of = [&](bool act) { return act ? (wk.k_end - wk.k_begin + C::kStageK - 1) / C::kStageK : 0; };

  // ------------------------------------------------------------------ prologue
  // The producer (MoE: after resolving the work -- gate_up's routed CTAs wait
  // for the router there) initialises the barriers and starts the weights.
  if constexpr (!kDense) {
    if (warp == C::kProducerWarp) resolve_work<kMode, kNT>(p, *mwork, 0, lane);
  }
  if (warp == C::kProducerWarp && lane == 0) {
    prefetch_tensormap(&p.tm_w);
    if constexpr (kDense) prefetch_tensormap(&p.tm_x);
    else prefetch_tensormap(&p.tm_w2);
    s_abort = 0;
    s_last = 0;
    bool act = true;
    int ntok0 = p.M;
    if constexpr (!kDense) {
      copy_work(*mwork, wk);
      act = mwork->active != 0;
      ntok0 = act ? mwork->ntok : 0;
    }
    // arrivals: dense, the producer (+ the converter on the f16 route); MoE,
    // the 32 gathering lanes' cp.async and lane 0 (the f16 route moves the
    // 32 to bar_xfull and adds the converter)
    const bool f16 = !kCoop && C::kHasF16 && ntok0 <= C::kF16MaxM;  // (converter warp)
    for (int i = 0; i < nstages; ++i) {
      mbar_init(smem_u32(&bar_full[i]), f16 ? 2 : (kDense ? 1 : 33));
      mbar_init(smem_u32(&bar_empty[i]), cw);
      mbar_init(smem_u32(&bar_xfull[i]), kDense ? 1 : 32);
      s_xbad[i] = -1;
    }
    mbar_init(smem_u32(&bar_inbox), 1);
    if (S > 1) {
      const int u = unit_of(), r = (u + static_cast<int>(S) - 1) / static_cast<int>(S);
      const int mine0 = max(0, min(r, u - static_cast<int>(rank) * r)) * rpf_of();
      mbar_arrive_expect_tx(smem_u32(&bar_inbox), S * ntok0 * mine0 * 4);  // tokens < ntok only
    }
    mbar_fence_init();
    const int pre0 = min(stages_of(act), nstages);
    for (int s = 0; s < pre0; ++s)
      if (!kDense || s != p.skip_stage) issue_weights(s, s);
  }
  __syncthreads();
  if (S > 1) cluster_arrive_relaxed();  // paired with a wait before the first remote access
  if (tid == 0) pdl_launch_dependents();
  bool active = true;
  int ntok = p.M;  // valid B rows (tokens, or pairs of the expert chunk)
  if constexpr (!kDense) {
    copy_work(*mwork, wk);
    active = mwork->active != 0;
    ntok = active ? mwork->ntok : 0;
  }
  const int nst = stages_of(active);
  const int pre = min(nst, nstages);
  const int unit = unit_of();
  const int R = (unit + static_cast<int>(S) - 1) / static_cast<int>(S);
  const int f_lo = static_cast<int>(rank) * R;
  const int f_hi = min(unit, f_lo + R);
  const int rpf = rpf_of();  // rows per feature
  const int mine = max(0, f_hi - f_lo) * rpf;
  const bool f16route = !kCoop && C::kHasF16 && ntok <= C::kF16MaxM;  // converter-warp f16 route
  // kF16MaxM < ntok <= 12: the consumer warps convert each stage's
  // activations to f16 together (one to three 16-byte chunks per thread) and
  // agree on exactness at a barrier; one converter warp would not keep up.
  const bool coop = kCoop;  // (the host launches this variant from 3 tokens)
  const bool f16acc = f16route || coop;  // acc holds exact f16-route products

  float acc[kChains][C::kTiles][4];  // main route's stages
  float accb[kF16 ? C::kTiles : 1][4];  // f16 route: fallback stages (bf16, products times 2^-kShift)
#pragma unroll
  for (int t = 0; t < C::kTiles; ++t) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
#pragma unroll
      for (int q = 0; q < kChains; ++q) acc[q][t][e] = 0.0f;
    }
  }
#pragma unroll
  for (int t = 0; t < (kF16 ? C::kTiles : 1); ++t) accb[t][0] = accb[t][1] = accb[t][2] = accb[t][3] = 0.0f;
  const int g = lane / 4, c = lane % 4;
  const int sg = (g % 2) * 4 + g / 2;  // sigma(g)
  const int row0 = warp * 16 + sg;     // tile rows of MMA rows g and g + 8
  const int row1 = row0 + 8;

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------------ producer
    pdl_wait();
    if constexpr (kDense) {
      if (lane == 0) {
        for (int s = 0, slot = 0, ph = 0; s < nst && !s_abort; ++s, slot = slot + 1 == nstages ? 0 : slot + 1, ph ^= slot == 0) {
          const uint32_t st = ring + slot * p.stage_bytes;
          const uint32_t fb = smem_u32(&bar_full[slot]);
          if (s >= pre && !mbar_wait_sleepy(smem_u32(&bar_empty[slot]), ph ^ 1, p.err, 64)) { s_abort = 1; break; }
          // (test hook: nothing at all for the skipped stage -- no copy and no
          // arrival, so the consumers' wait for it runs out with nothing in flight)
          if (s == p.skip_stage) continue;
          if (s >= pre) issue_weights(s, slot);
          const int k0 = wk.k_begin + s * C::kStageK;
          if (f16route) {
            const uint32_t xb = smem_u32(&bar_xfull[slot]);
            mbar_arrive_expect_tx(xb, C::kXBytes);
            tma_load_3d(st + p.x_off, &p.tm_x, 0, 0, k0 / kSubK, xb, pol_x);
            mbar_arrive(fb);
          } else {
            mbar_arrive_expect_tx(fb, C::kXBytes);
            tma_load_3d(st + p.x_off, &p.tm_x, 0, 0, k0 / kSubK, fb, pol_x);
          }
        }
      }
    } else {
      // Gathered activations: lane c copies 16-byte chunk c (of 32) of every
      // B row of the stage into the 128-byte-swizzled atoms (rows past the
      // chunk's pairs / tokens are zero-filled).
      const uint16_t* xb = wk.shared ? p.x2 : p.x;
      const int u = lane / 8, cc = lane % 8;
      for (int s = 0, slot = 0, ph = 0; s < nst && !s_abort; ++s, slot = slot + 1 == nstages ? 0 : slot + 1, ph ^= slot == 0) {
        const uint32_t st = ring + slot * p.stage_bytes;
        const uint32_t fb = smem_u32(&bar_full[slot]);
        if (s >= pre) {
          const bool ok =
              __all_sync(0xFFFFFFFFu, mbar_wait_sleepy(smem_u32(&bar_empty[slot]), ph ^ 1, p.err, 64));
          if (!ok) { s_abort = 1; break; }
          if (lane == 0) issue_weights(s, slot);
          __syncwarp();
        }
        const int k0 = wk.k_begin + s * C::kStageK;
        const bool kok = lane * 8 < min(C::kStageK, wk.k_end - k0);
        const uint16_t* src_k = xb + k0 + lane * 8;
        const uint32_t dst0 = st + p.x_off + u * (kNT * 128);
#pragma unroll
        for (int n = 0; n < kNT; ++n) {
          const bool valid = kok && n < ntok;
          const uint32_t dst = dst0 + (n / 8) * 1024 + (n % 8) * 128 + ((cc ^ (n % 8)) * 16);
          cp_async16(dst, valid ? src_k + mwork->xoff[n] : xb, valid ? 16u : 0u);
        }
        cp_async_arrive_noinc(f16route ? smem_u32(&bar_xfull[slot]) : fb);
        if (lane == 0) mbar_arrive(fb);
      }
    }
  } else if (warp == C::kConverterWarp) {
    // ------------------------------------------------------------------ converter
    if (f16route)
    // Rows < ntok of each stage's activations to f16 in place (16-byte
    // chunks); the other rows and K past the end are zero-filled, the same bits
    // in f16.  A stage with any inexact value is flagged for the bf16 route.
    for (int s = 0, slot = 0, ph = 0; s < nst; ++s, slot = slot + 1 == nstages ? 0 : slot + 1, ph ^= slot == 0) {
      const uint32_t st = ring + slot * p.stage_bytes;
      const bool ok = __all_sync(0xFFFFFFFFu, !s_abort && mbar_wait(smem_u32(&bar_xfull[slot]), ph, p.err));
      if (!ok) {
        s_abort = 1;
        break;
      }
      const int kvalid = min(C::kStageK, wk.k_end - wk.k_begin - s * C::kStageK);
      bool exact = true;
      for (int id = lane; id < ntok * 32; id += 32) {
        const int n = id / 32, q = id % 32;
        if (8 * q >= kvalid) continue;
        const uint32_t a = st + p.x_off + (q / 8) * (kNT * 128) + (n / 8) * 1024 + (n % 8) * 128 +
                           ((static_cast<uint32_t>(q % 8) ^ static_cast<uint32_t>(n % 8)) * 16);
        const uint4 v = lds128(a);
        uint4 o;
        exact &= bf16x2_to_f16x2_exact(v.x, o.x);
        exact &= bf16x2_to_f16x2_exact(v.y, o.y);
        exact &= bf16x2_to_f16x2_exact(v.z, o.z);
        exact &= bf16x2_to_f16x2_exact(v.w, o.w);
        sts128(a, o);
      }
      if (!__all_sync(0xFFFFFFFFu, exact) && lane == 0) s_xbad[slot] = s;
      fence_proxy_async_smem();  // these writes precede the slot's next TMA fill
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_full[slot]));
    }
  } else {
    // ------------------------------------------------------------------ consumers
    // shared-memory offsets of this thread's two rows (128-byte swizzle key
    // = row % 8, the same for both rows) and of their scale bytes
    const uint32_t key = static_cast<uint32_t>(row0 % 8);
    const uint32_t w_off0 = (row0 / 8) * 1024 + (row0 % 8) * 128;
    const uint32_t w_off1 = (row1 / 8) * 1024 + (row1 % 8) * 128;
    // (static indices only, so the work description stays in registers)
    auto sf_off = [&](int row) -> uint32_t {
      const int half = trows / 2;
      const bool b1 = wk.paired && row >= half;
      const int r = (b1 ? wk.srow[1] : wk.srow[0]) + (b1 ? row - half : row);
      // stage slot of r's group: the valid groups are stored in order
      const int g = r / 128;
      const int gslot = b1 ? (wk.sgroup[0] >= 0) + (wk.sgroup[1] >= 0) + (g != wk.sgroup[2]) : (g != wk.sgroup[0]);
      return trows * 128 + gslot * 2048 + (r % 32) * 16 + ((r % 128) / 32) * 4;
    };
    const uint32_t sf0 = sf_off(row0), sf1 = sf_off(row1);
    // global activation rows of this thread's B rows (f16 route's fallback)
    const uint16_t* xrow[C::kTiles];
#pragma unroll
    for (int t = 0; t < C::kTiles; ++t) {
      const int n = 8 * t + g;
      if constexpr (kDense) xrow[t] = n < ntok ? p.x + static_cast<int64_t>(n) * p.ldx : nullptr;
      else xrow[t] = n < ntok ? (wk.shared ? p.x2 : p.x) + mwork->xoff[n] : nullptr;
    }
    // B rows (tokens) past ntok are zero in the stage; lanes holding them use
    // zero registers instead of loading (the same products, less shared-memory
    // traffic: at M = 1 only a quarter warp loads activations).
    // One 128-K half of a stage: chunk j = 4 h + c of both rows.  `cvalid`
    // false (a chunk past the end of a ragged last stage) gives zero A
    // registers: that chunk's scales were not copied and may hold anything.
    auto half_f16 = [&](uint32_t st, int h, bool cvalid) {
      const int j = 4 * h + c;
      const uint4 A0 = lds128(st + w_off0 + ((static_cast<uint32_t>(j) ^ key) * 16));
      const uint4 A1 = lds128(st + w_off1 + ((static_cast<uint32_t>(j) ^ key) * 16));
      const uint32_t sc_off = (j / 2) * 512 + 2 * (j % 2);
      uint32_t s0lo, s0hi, s1lo, s1hi;
      scale_pair_to_f16x2(lds16(st + sf0 + sc_off), s0lo, s0hi);
      scale_pair_to_f16x2(lds16(st + sf1 + sc_off), s1lo, s1hi);
      if (!cvalid) s0lo = s0hi = s1lo = s1hi = 0u;
      const uint32_t a0w[4] = {A0.x, A0.y, A0.z, A0.w};
      const uint32_t a1w[4] = {A1.x, A1.y, A1.z, A1.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t r0[4], r1[4];
        dequant8_f16(a0w[w], w < 2 ? s0lo : s0hi, r0);
        dequant8_f16(a1w[w], w < 2 ? s1lo : s1hi, r1);
        // the f16 activations of the same 8 K (natural order): atom u, chunk ch
        const int kk = 32 * j + 8 * w;
        const uint32_t u = kk / 64, ch = (kk % 64) / 8;
#pragma unroll
        for (int t = 0; t < C::kTiles; ++t) {
          const int n = 8 * t + g;
          const uint4 xv = lds128_if(st + p.x_off + u * (kNT * 128) + (n / 8) * 1024 + (n % 8) * 128 +
                                         ((ch ^ static_cast<uint32_t>(n % 8)) * 16),
                                     n < ntok);
          mma_f16_16816(acc[(2 * w) % kChains][t], r0[0], r1[0], r0[1], r1[1], xv.x, xv.y);
          mma_f16_16816(acc[(2 * w + 1) % kChains][t], r0[2], r1[2], r0[3], r1[3], xv.z, xv.w);
        }
      }
    };
    // bf16 route, activations from the stage in shared memory (permuted in
    // registers to the weight pairs' K order)
    auto half_bf16_smem = [&](uint32_t st, int h, bool cvalid) {
      const int j = 4 * h + c;
      const uint4 A0 = lds128(st + w_off0 + ((static_cast<uint32_t>(j) ^ key) * 16));
      const uint4 A1 = lds128(st + w_off1 + ((static_cast<uint32_t>(j) ^ key) * 16));
      const uint32_t sc_off = (j / 2) * 512 + 2 * (j % 2);
      uint32_t s0lo, s0hi, s1lo, s1hi;
      scale_pair_to_bf16x2(lds16(st + sf0 + sc_off), s0lo, s0hi);
      scale_pair_to_bf16x2(lds16(st + sf1 + sc_off), s1lo, s1hi);
      if (!cvalid) s0lo = s0hi = s1lo = s1hi = 0u;
      const uint32_t a0w[4] = {A0.x, A0.y, A0.z, A0.w};
      const uint32_t a1w[4] = {A1.x, A1.y, A1.z, A1.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t r0[4], r1[4];
        e2m1x8_raw_perm(a0w[w], r0);
        e2m1x8_raw_perm(a1w[w], r1);
        const uint32_t sa = w < 2 ? s0lo : s0hi, sb = w < 2 ? s1lo : s1hi;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          r0[q] = bf16x2_mul(r0[q], sa);
          r1[q] = bf16x2_mul(r1[q], sb);
        }
        const int kk = 32 * j + 8 * w;
        const uint32_t u = kk / 64, ch = (kk % 64) / 8;
#pragma unroll
        for (int t = 0; t < C::kTiles; ++t) {
          const int n = 8 * t + g;
          const uint4 xv = perm_x8(lds128_if(st + p.x_off + u * (kNT * 128) + (n / 8) * 1024 + (n % 8) * 128 +
                                                 ((ch ^ static_cast<uint32_t>(n % 8)) * 16),
                                             n < ntok));
          mma_bf16_16816(acc[(2 * w) % kChains][t], r0[0], r1[0], r0[1], r1[1], xv.x, xv.y);
          mma_bf16_16816(acc[(2 * w + 1) % kChains][t], r0[2], r1[2], r0[3], r1[3], xv.z, xv.w);
        }
      }
    };
    // bf16 route with the activations from global memory: the f16 route's
    // fallback for a stage whose activations are not all exact f16
    auto half_bf16 = [&](uint32_t st, int k0, int h, bool cvalid) {
      const int j = 4 * h + c;
      const uint4 A0 = lds128(st + w_off0 + ((static_cast<uint32_t>(j) ^ key) * 16));
      const uint4 A1 = lds128(st + w_off1 + ((static_cast<uint32_t>(j) ^ key) * 16));
      const uint32_t sc_off = (j / 2) * 512 + 2 * (j % 2);
      uint32_t s0lo, s0hi, s1lo, s1hi;
      scale_pair_to_bf16x2(lds16(st + sf0 + sc_off), s0lo, s0hi);
      scale_pair_to_bf16x2(lds16(st + sf1 + sc_off), s1lo, s1hi);
      if (!cvalid) s0lo = s0hi = s1lo = s1hi = 0u;
      const uint32_t a0w[4] = {A0.x, A0.y, A0.z, A0.w};
      const uint32_t a1w[4] = {A1.x, A1.y, A1.z, A1.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t r0[4], r1[4];
        e2m1x8_raw_perm(a0w[w], r0);
        e2m1x8_raw_perm(a1w[w], r1);
        const uint32_t sa = w < 2 ? s0lo : s0hi, sb = w < 2 ? s1lo : s1hi;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          r0[q] = bf16x2_mul(r0[q], sa);
          r1[q] = bf16x2_mul(r1[q], sb);
        }
        // the original bf16 activations of the same 8 K, from global memory
        const int kk = 32 * j + 8 * w;
#pragma unroll
        for (int t = 0; t < C::kTiles; ++t) {
          uint4 xv = make_uint4(0u, 0u, 0u, 0u);
          if (cvalid && xrow[t] != nullptr) xv = perm_x8(__ldg(reinterpret_cast<const uint4*>(xrow[t] + k0 + kk)));
          mma_bf16_16816(accb[kF16 ? t : 0], r0[0], r1[0], r0[1], r1[1], xv.x, xv.y);
          mma_bf16_16816(accb[kF16 ? t : 0], r0[2], r1[2], r0[3], r1[3], xv.z, xv.w);
        }
      }
    };
    // Cooperative f16 conversion of a stage's activation rows < ntok (the
    // consumer warps' threads take chunks round-robin), then a barrier that
    // ORs "inexact or gave up" over them: 0 = every value exact (f16 route),
    // 1 = some value inexact (bf16 fallback), 2 = a warp's wait gave up (all
    // leave the loop).  A thread whose wait gave up still joins, so no warp is
    // left at the barrier, and the decision to leave comes from the barrier,
    // the same for every warp.
    auto coop_convert = [&](uint32_t st, int kvalid, bool gave_up) -> int {
      bool bad = gave_up;
      if (!gave_up) {
        for (int id = warp * 32 + lane; id < ntok * 32; id += cw * 32) {
          const int n = id / 32, q = id % 32;
          if (8 * q >= kvalid) continue;
          const uint32_t a = st + p.x_off + (q / 8) * (kNT * 128) + (n / 8) * 1024 + (n % 8) * 128 +
                             ((static_cast<uint32_t>(q % 8) ^ static_cast<uint32_t>(n % 8)) * 16);
          const uint4 v = lds128(a);
          uint4 o;
          bool exact = bf16x2_to_f16x2_exact(v.x, o.x);
          exact &= bf16x2_to_f16x2_exact(v.y, o.y);
          exact &= bf16x2_to_f16x2_exact(v.z, o.z);
          exact &= bf16x2_to_f16x2_exact(v.w, o.w);
          sts128(a, o);
          bad |= !exact;
        }
        fence_proxy_async_smem();  // these writes precede the slot's next TMA fill
      }
      if (!bar_red_or<2>(cw * 32, bad)) return 0;
      return bar_red_or<2>(cw * 32, gave_up) ? 2 : 1;  // (every thread takes this branch or none)
    };
    // (warps past cw own no rows of this tile: they skip the stream)
    for (int s = 0, slot = 0, ph = 0; s < (warp < cw ? nst : 0);
         ++s, slot = slot + 1 == nstages ? 0 : slot + 1, ph ^= slot == 0) {
      const uint32_t st = ring + slot * p.stage_bytes;
      const bool ok = __all_sync(0xFFFFFFFFu, !s_abort && mbar_wait(smem_u32(&bar_full[slot]), ph, p.err));
      if (!ok) s_abort = 1;
      // valid K of the stage: 64 .. 256 in steps of 64; a chunk (32 K) is
      // wholly valid or wholly past the end, where its A registers are zero
      // (its scales were not copied and may hold anything)
      const int kvalid = min(C::kStageK, wk.k_end - wk.k_begin - s * C::kStageK);
      bool use_f16 = false;
      if (coop) {
        const int r = coop_convert(st, kvalid, !ok);
        if (r == 2) break;
        use_f16 = r == 0;
      } else if (!ok) {
        break;
      } else if (f16route) {
        use_f16 = s_xbad[slot] != s;  // bar_full included the converter's arrival
      }
      if (!f16acc) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (128 * h < kvalid) {
            if (128 * (h + 1) <= kvalid) half_bf16_smem(st, h, true);
            else half_bf16_smem(st, h, 32 * (4 * h + c) < kvalid);
          }
        }
      } else if constexpr (kF16) {
        if (use_f16) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (128 * h < kvalid) {
              if (128 * (h + 1) <= kvalid) half_f16(st, h, true);
              else half_f16(st, h, 32 * (4 * h + c) < kvalid);
            }
          }
        } else {
          pdl_wait();  // the activations are read from global memory directly
          const int k0 = wk.k_begin + s * C::kStageK;
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            if (128 * h < kvalid) half_bf16(st, k0, h, 32 * (4 * h + c) < kvalid);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar_empty[slot]));
    }
  }

  // ==================================================================== epilogue
  __syncwarp();
  if (warp < C::kConsumerWarps) {
    const float post = static_cast<float>(1 << kShift);
    // Push this thread's partials (rows row0 / row1, tokens 8t + 2c + {0,1}
    // below ntok) to the owners of the rows: inbox[src][n][rr].
    if (S > 1) cluster_wait();  // all peers' inbox barriers are initialised
    const bool go = !s_abort;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      if (warp >= cw) break;  // (rows past the tile)
      const int row = hr ? row1 : row0;
      const int fi = row % unit;
      const int owner = fi / R;
      const int owner_feats = min(R, unit - owner * R);
      const int rr = (row / unit) * owner_feats + (fi - owner * R);
      const int rows_owner = owner_feats * rpf;
      const uint32_t base = inbox + ((rank * kNT) * rows_owner + rr) * 4;
      const uint32_t rbase = S > 1 ? mapa(base, static_cast<uint32_t>(owner)) : base;
      const uint32_t rbar = S > 1 ? mapa(smem_u32(&bar_inbox), static_cast<uint32_t>(owner)) : 0u;
#pragma unroll
      for (int t = 0; t < C::kTiles; ++t) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int n = 8 * t + 2 * c + e;
          float a16 = 0.0f;
#pragma unroll
          for (int q = 0; q < kChains; ++q) a16 += acc[q][t][2 * hr + e];
          // acc holds the main route's products (exact on the f16 route,
          // times 2^-kShift on the bf16 route); accb the f16 route's fallback
          if (!f16acc) a16 *= post;
          if constexpr (kF16) a16 += accb[t][2 * hr + e] * post;
          const float v = go ? a16 : 0.0f;
          const uint32_t off = n * rows_owner * 4;
          if (n >= ntok) continue;
          if (S > 1) st_async_f32(rbase + off, v, rbar);
          else stsf(rbase + off, v);
        }
      }
    }
    if (S > 1) {
      if (!mbar_wait<true>(smem_u32(&bar_inbox), 0, p.err)) s_abort = 1;
    } else {
      epi_sync<kEpiThreads>();
    }
    auto partial = [&](int n, int lr) -> float {
      float a = 0.0f;
      for (uint32_t src = 0; src < S; ++src) a += ldsf(inbox + ((src * kNT + n) * mine + lr) * 4);
      return a;
    };
    const int nf = f_hi - f_lo;
    if (active && !s_abort && nf > 0) {
      pdl_wait();
      if (rpf == 1) {
        // plain tiles: feature = tile row (dense out, or the down y scratch)
        float sc = 1.0f;
        uint16_t* dst = p.out;
        int64_t ld = p.ldo;
        int nfeat = p.n_out;
        if constexpr (kDense) {
          sc = __ldg(p.gs);
        } else {
          sc = wk.shared ? __ldg(p.gs) : __ldg(p.alpha + wk.expert);
          if (wk.shared) {
            dst = p.out2;
            ld = p.ldo2;
            nfeat = p.shared_n_out;
          }
        }
        for (int it = tid; it < nf * ntok; it += kEpiThreads) {
          const int n = it / nf, lr = it % nf;
          const int o = wk.out_base + f_lo + lr;
          if (o >= nfeat) continue;
          const int64_t orow = kDense ? n : mwork->orow[n];
          dst[orow * ld + o] = f32_to_bf16_rn(partial(n, lr) * sc);
        }
      } else if (kMode == kMoeGateUp && !wk.shared) {
        // routed [up; gate] group: feature o = up row o, gate row o + 64
        const float al = __ldg(p.alpha + wk.expert);
        for (int it = tid; it < nf * ntok; it += kEpiThreads) {
          const int n = it / nf, lr = it % nf;
          const int feat = wk.out_base + f_lo + lr;
          if (feat >= p.n_out) continue;
          const float uu = partial(n, lr) * al;
          const float gt = partial(n, lr + nf) * al;
          p.out[static_cast<int64_t>(mwork->orow[n]) * p.ldo + feat] = f32_to_bf16_rn(silu_fast(gt) * uu);
        }
      } else {
        // paired tiles: feature o = gate row o, up row o + 64
        const float gs = __ldg(p.gs);
        uint16_t* dst = kDense ? p.out : p.out2;
        const int64_t ld = kDense ? p.ldo : p.ldo2;
        const int nfeat = kDense ? p.n_out : p.shared_n_out;
        for (int it = tid; it < nf * ntok; it += kEpiThreads) {
          const int n = it / nf, lr = it % nf;
          const int feat = wk.out_base + f_lo + lr;
          if (feat >= nfeat) continue;
          const float G = bf16_to_f32(f32_to_bf16_rn(partial(n, lr) * gs));
          const float U = bf16_to_f32(f32_to_bf16_rn(partial(n, lr + nf) * gs));
          const int64_t orow = kDense ? n : mwork->orow[n];
          dst[orow * ld + feat] = f32_to_bf16_rn(silu_exact(G) * U);
        }
      }
    }
    if constexpr (kMode == kMoeDown) {
      // Every CTA of a row-tile column arrives once (tagged with this call's
      // epoch, so the scratch needs no zero-fill); the last one combines:
      // out[t] = bf16(bf16(sum_j tw[t, j] * y[t, j]) + y_shared[t]).
      epi_sync<kEpiThreads>();
      if (tid == 0) {
        // The previous grid in the stream may be a down_combine on the same
        // workspace (PDL lets this grid start early): its counting must be
        // over before this call's first arrival, which retags the counter.
        pdl_wait();
        __threadfence();
        unsigned long long* ctr = p.counters + blockIdx.x;
        const unsigned long long tag = static_cast<unsigned long long>(p.epoch) << 32;
        unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(ctr), next;
        for (;;) {
          next = ((old & 0xFFFFFFFF00000000ull) == tag) ? old + 1 : tag + 1;
          const unsigned long long seen = atomicCAS(ctr, old, next);
          if (seen == old) break;
          old = seen;
        }
        s_last = static_cast<uint32_t>(next) == gridDim.y;
        if (s_last) atomicExch(ctr, 0ull);
        __threadfence();
      }
      epi_sync<kEpiThreads>();
      if (s_last) {
        pdl_wait();
        moe_combine_tile<kOcc >= 3 ? 2 : 8>(p, blockIdx.x * 128, tid, kEpiThreads);  // (64 registers at three CTAs per SM)
      }
    }
  } else if (S > 1) {
    cluster_wait();  // the producer warp closes its cluster-barrier phase
  }
  __syncthreads();
}

}  // namespace fp4
