// k_gemv.cuh -- the small-M GEMV pipeline on tcgen05 tensor cores.
//
// One kernel template serves the dense NVFP4 GEMV (optionally with the fused
// silu_mul epilogue), the BF16-weight GEMV, and both MoE kernels
// (vllm.models.flint.ops.nvfp4_gemv nvfp4_gemv / bf16_gemv,
// vllm.models.flint.ops.moe_gemv gate_up / down_combine).
//
// Swap-AB: a CTA owns kT tiles of 128 weight rows (the MMA M dimension); the
// tokens are the MMA N dimension (kNT = 16 .. 128).  Its K range is a slice
// of K; the kS CTAs of a cluster split K and reduce their fp32 partials
// through distributed shared memory in rank order (deterministic).
//
// Warp roles (kT dequant warpgroups, then one producer and one MMA warp):
//   producer  lane 0 streams weight tiles (TMA, 128-byte swizzle) and the
//             matching 512-byte scale chunks (bulk copies) into a ring of
//             shared-memory stages; with PDL these loads are issued before
//             griddepcontrol.wait.  All 32 lanes then copy the activation
//             rows of each stage with cp.async (after the wait).
//   dequant   warpgroup t: thread i owns row i of tile t.  Per 64-wide K
//             slice it reads 32 code bytes and 4 scale bytes, dequantizes
//             them exactly to bf16 (dequant.cuh) and stores them with
//             tcgen05.st into a tensor-memory A slot.  Warpgroup 0 also
//             permutes the activation slice in shared memory to the weight
//             pairs' K order.
//   mma       one thread issues tcgen05.mma (A from tensor memory, B = the
//             activations from shared memory, fp32 D in tensor memory) and
//             frees A slots / ring stages with tcgen05.commit.
//   epilogue  the dequant warpgroups read D with tcgen05.ld, exchange
//             partials through (distributed) shared memory and apply the
//             mode's epilogue.
// The BF16-weight mode has no dequant step: both operands come from shared
// memory by TMA (tcgen05.mma with two smem descriptors).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "dequant.cuh"

namespace fp4 {

enum Mode : int {
  kDenseFp4 = 0,   // nvfp4_gemv; kT = 2 fuses silu_mul ([gate | up] halves)
  kDenseBf16 = 1,  // bf16_gemv and the GEMM of the dequantize + GEMM path
  kMoeGateUp = 2,  // routed experts ([up; gate] 64-row groups) + shared expert
  kMoeDown = 3,    // routed + shared experts into scratch, last CTA combines
};

constexpr int kMaxStages = 8;
constexpr int kSlots = 4;       // tensor-memory A slots (default)
constexpr int kMaxSlots = 8;
constexpr int kSubK = 64;       // K per A slot / per activation atom
constexpr int kStageK4 = 256;   // K per ring stage, NVFP4 weights (128 B per row)
constexpr int kStageK16 = 64;   // K per ring stage, bf16 weights (128 B per row)
constexpr int kMaxNT = 128;

struct GemvParams {
  CUtensorMap tm_w;    // weights read by routed / dense CTAs
  CUtensorMap tm_w2;   // shared-expert weights (MoE)
  CUtensorMap tm_x;    // bf16 mode: activations [M, K], box {64, kNT}
  const uint8_t* sf;   // scales of tm_w rows (MoE: E consecutive buffers)
  const uint8_t* sf2;  // scales of tm_w2 rows
  const uint16_t* x;   // activations (bf16 bits) of routed / dense CTAs
  const uint16_t* x2;  // activations of shared-expert CTAs
  int64_t ldx, ldx2;
  const float* gs;     // dense global scale / shared-expert global scale
  const float* alpha;  // MoE per-expert scale
  const int32_t* ids;  // MoE expert ids [M, topk]
  const float* tw;     // MoE top-k weights [M, topk]
  uint16_t* out;       // dense out / gate_up act / down y scratch
  int64_t ldo;
  uint16_t* out2;      // gate_up sact / down y_shared scratch
  int64_t ldo2;
  uint16_t* out3;      // down: final output [M, H]
  unsigned long long* counters;  // down: per row-tile arrival counters [epoch:32 | count:32]
  uint32_t epoch;      // down: nonzero tag of this call (counters from other calls read as 0)
  int M;               // tokens
  int n_out;           // dense: output features; MoE routed: output features
  int n_half;          // dense silu: N / 2 (first up row); shared gate_up: SI
  int K;               // dense / routed K
  int K2;              // shared-expert K
  int k_split;         // dense: K elements per cluster rank (multiple of 64)
  int E, topk, P;      // MoE (P = M * topk)
  int rows_per_expert; // MoE routed weight rows per expert
  int rows_w;          // rows of the dense / shared weight (scale groups)
  int shared_n_out;    // MoE shared output features
  int routed_tiles;    // MoE: column tiles per routed expert
  int shared_tiles;    // MoE: column tiles of the shared expert
  int kbp, kbp2;       // padded K blocks (K/16 rounded up to 4) of tm_w / tm_w2 rows
  uint32_t sf_expert_bytes;
  int nstages;
  uint32_t* err;       // device error word
};

struct CtaWork {
  int active;      // 0: nothing to compute
  int shared;      // 1: shared-expert CTA (MoE)
  int ntok;        // valid B rows
  int k_begin, k_end;
  int wrow[2];     // tensor-map row of each tile's first row
  int srow[2];     // first row in the scale buffer's row space
  int sgroups[2];  // 128-row scale groups to copy per tile (0..2)
  int kbp;
  int expert;
  int out_base;    // first output feature of tile 0
  float scale;     // alpha[e] or the global scale (loaded after the PDL wait)
  int tok[kMaxNT];   // B row -> activation row
  int orow[kMaxNT];  // B row -> output row (pair / token)
  long long xoff[kMaxNT];  // B row -> element offset of its activation row
};

__host__ __device__ constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p *= 2;
  return p;
}

template <int kMode, int kT, int kNT>
struct Cfg {
  static constexpr bool kFp4 = kMode != kDenseBf16;
  // Dequant warpgroups per tile: the G warpgroups of a tile take turns on
  // consecutive 64-wide K slices, so G slices of a tile are in flight.
  static constexpr int kG = kFp4 ? 2 : 1;
  static constexpr int kWarpgroups = kT * kG;
  static constexpr int kWarps = 4 * kWarpgroups + 2;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kProducerWarp = 4 * kWarpgroups;
  static constexpr int kMmaWarp = 4 * kWarpgroups + 1;
  static constexpr int kStageK = kFp4 ? kStageK4 : kStageK16;
  static constexpr int kWTileBytes = 128 * 128;
  static constexpr int kSfTileBytes = kFp4 ? 2 * 4 * 512 : 0;
  static constexpr int kXBytes = kNT * kStageK * 2;
  static constexpr int kXOff = kT * (kWTileBytes + kSfTileBytes);
  static constexpr int kStageBytes = kXOff + kXBytes;
  // Tensor memory: A slots (64 K each, fp4 modes) and kAcc independent fp32
  // accumulators per tile.  Consecutive K=16 MMAs of a slice go to different
  // accumulators so they do not serialise on one accumulator; the epilogue
  // sums them.  Sized to 256 columns (two CTAs per SM) for one tile, 512 for
  // two.
  static constexpr int kSlotsUsed = (kT == 2 && kNT <= 16) ? 6 : kSlots;
  static constexpr int kTmemA = kFp4 ? kSlotsUsed * kT * 32 : 0;
  static constexpr int kBudget = kT == 1 ? 256 : 512;
  static constexpr int kAcc = kTmemA + 4 * kT * kNT <= kBudget ? 4 : kTmemA + 2 * kT * kNT <= kBudget ? 2 : 1;
  static constexpr int kTmemCols = pow2_at_least(kTmemA + kAcc * kT * kNT);
  static constexpr int kRedBytes = kT * kNT * 128 * 4;
  // Dense modes read contiguous activation rows with TMA; the MoE modes
  // gather rows by token / pair with cp.async from the producer lanes.
  static constexpr bool kXTma = kMode == kDenseFp4 || kMode == kDenseBf16;
  static constexpr int kFullCount = kXTma ? 1 : 33;
  // Split-K partials are pushed to the owning cluster rank (st.async into a
  // dedicated inbox) when the inbox is small; otherwise pulled through DSMEM
  // from the (reused) ring.
  static constexpr bool kPush = kT * kNT <= 64;
  static constexpr int kInboxBytes = kPush ? kT * kNT * 136 * 4 : 0;
  static_assert(kNT % 16 == 0 && kNT >= 16 && kNT <= kMaxNT, "token tile");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kTmemCols <= 512, "tensor memory");
  static_assert(kSlotsUsed <= kMaxSlots, "slot barriers");
  // CTAs per SM the launch aims for (tensor memory is 512 columns per SM)
  static constexpr int kMinBlocks = kTmemCols <= 256 ? 2 : 1;
};

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// SiLU with IEEE exp and division (the "exact" SiLU of the dense path).
__device__ __forceinline__ float silu_exact(float g) { return __fdiv_rn(g, 1.0f + expf(-g)); }
// SiLU with the fast exponential and division (the routed experts' fast sigmoid).
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Named barrier over the epilogue (dequant) warpgroups only.
template <int kThreadsEpi>
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreadsEpi) : "memory");
}

// Eight columns [c, c+8) of a tile's accumulator: the sum of its kAcc
// partial accumulators (kNT columns apart) in tensor memory.
template <int kAcc, int kNT>
__device__ __forceinline__ void load_acc(uint32_t taddr, float (&out)[8]) {
  uint32_t v[8];
  tmem_ld8(taddr, v);
  tmem_wait_ld();
#pragma unroll
  for (int j = 0; j < 8; ++j) out[j] = __uint_as_float(v[j]);
#pragma unroll
  for (int a = 1; a < kAcc; ++a) {
    tmem_ld8(taddr + a * kNT, v);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 8; ++j) out[j] += __uint_as_float(v[j]);
  }
}

// Resolve what this CTA computes (thread 0).  Returns false if the ids could
// not be read yet (gate_up routed: caller waits for the previous grid first).
template <int kMode, int kT, int kNT>
__device__ void resolve_work(const GemvParams& p, CtaWork& w, uint32_t split) {
  w.active = 1;
  w.shared = 0;
  w.expert = -1;
  w.scale = 1.0f;
  w.sgroups[0] = w.sgroups[1] = 0;
  w.wrow[1] = w.srow[1] = 0;
  const int tile = blockIdx.x / max(1u, cluster_nctarank());
  if constexpr (kMode == kDenseFp4 || kMode == kDenseBf16) {
    w.ntok = p.M;  // B row n is token n (activations read by TMA)
    w.k_begin = static_cast<int>(split) * p.k_split;
    w.k_end = min(p.K, w.k_begin + p.k_split);
    w.kbp = p.kbp;
    w.out_base = tile * 128;
    w.wrow[0] = tile * 128;
    if (kT == 2) w.wrow[1] = p.n_half + tile * 128;
    for (int t = 0; t < kT; ++t) {
      w.srow[t] = w.wrow[t];
      const int groups_total = (p.rows_w + 127) / 128;
      const int g0 = w.srow[t] / 128;
      const int g1 = min(w.srow[t] + 127, p.rows_w - 1) / 128;
      w.sgroups[t] = g0 < groups_total ? g1 - g0 + 1 : 0;
    }
  } else {
    // MoE: blockIdx.y < P: routed pair column; else shared-expert token chunk.
    const int col = blockIdx.y;
    w.k_begin = 0;
    if (col < p.P) {
      // gate_up runs right after the router: its ids are complete only after
      // the wait.  down_combine reads them early (they are two kernels old).
      if (kMode == kMoeGateUp) pdl_wait();
      const int e = __ldg(p.ids + col);
      if (tile >= p.routed_tiles) { w.active = 0; return; }
      if (e < 0 || e >= p.E) {
        raise_error(p.err, FP4_ERR_BADIDX);
        w.active = 0;
        return;
      }
      // rank of this pair among the pairs routed to e; the first pair of each
      // chunk of kNT pairs computes the whole chunk.
      int rank = 0;
      for (int q = 0; q < col; ++q) rank += (__ldg(p.ids + q) == e);
      if (rank % kNT != 0) { w.active = 0; return; }
      int n = 0;
      for (int q = col; q < p.P && n < kNT; ++q) {
        if (__ldg(p.ids + q) == e) {
          w.tok[n] = kMode == kMoeGateUp ? q / p.topk : q;  // x row (token) or act row (pair)
          w.orow[n] = q;
          ++n;
        }
      }
      w.ntok = n;
      for (; n < kNT; ++n) w.tok[n] = w.orow[n] = w.tok[0];
      w.expert = e;
      w.k_end = p.K;
      w.kbp = p.kbp;
      for (int t = 0; t < kT; ++t) {
        const int r0 = tile * 128 * kT + t * 128;  // row inside the expert
        w.wrow[t] = e * p.rows_per_expert + r0;
        w.srow[t] = r0;
        w.sgroups[t] = r0 < p.rows_per_expert ? 1 : 0;
      }
      w.out_base = tile * 128;
      for (int m = 0; m < kNT; ++m) w.xoff[m] = static_cast<long long>(w.tok[m]) * p.ldx;
    } else {
      const int chunk = col - p.P;
      if (tile >= p.shared_tiles) { w.active = 0; return; }
      w.shared = 1;
      const int t0 = chunk * kNT;
      w.ntok = min(kNT, p.M - t0);
      for (int n = 0; n < kNT; ++n) w.tok[n] = w.orow[n] = t0 + (n < w.ntok ? n : 0);
      w.k_end = p.K2;
      w.kbp = p.kbp2;
      w.wrow[0] = tile * 128;
      if (kT == 2) w.wrow[1] = p.n_half + tile * 128;
      for (int t = 0; t < kT; ++t) {
        w.srow[t] = w.wrow[t];
        const int groups_total = (p.rows_w + 127) / 128;
        const int g0 = w.srow[t] / 128;
        const int g1 = min(w.srow[t] + 127, p.rows_w - 1) / 128;
        w.sgroups[t] = g0 < groups_total ? g1 - g0 + 1 : 0;
      }
      w.out_base = tile * 128;
      for (int m = 0; m < kNT; ++m) w.xoff[m] = static_cast<long long>(w.tok[m]) * p.ldx2;
    }
  }
}

template <int kMode, int kT, int kNT>
__global__ void __launch_bounds__(Cfg<kMode, kT, kNT>::kThreads, Cfg<kMode, kT, kNT>::kMinBlocks)
    gemv_kernel(const __grid_constant__ GemvParams p) {
  using C = Cfg<kMode, kT, kNT>;
  constexpr int kEpiThreads = C::kWarpgroups * 128;
  constexpr int kG = C::kG;
  constexpr int kNS = C::kSlotsUsed;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-aligned ring, addressed through 32-bit shared-window addresses; the
  // split-K inbox (push mode) follows the ring.
  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t inbox = ring + p.nstages * C::kStageBytes;
  __shared__ __align__(8) uint64_t bar_full[kMaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t bar_afull[kMaxSlots];
  __shared__ __align__(8) uint64_t bar_aempty[kMaxSlots];
  __shared__ __align__(8) uint64_t bar_accum;
  __shared__ __align__(8) uint64_t bar_inbox;
  __shared__ __align__(8) uint64_t bar_red_ready;
  __shared__ __align__(8) uint64_t bar_red_done;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_last;
  __shared__ CtaWork s_work;

  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;
  const uint32_t S = cluster_nctarank();
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0;
  const int nstages = p.nstages;
  const int R = (128 + static_cast<int>(S) - 1) / static_cast<int>(S);  // rows reduced per cluster rank
  const int r_lo = static_cast<int>(rank) * R;
  const int r_hi = min(128, r_lo + R);

  // For gate_up the routed experts are only known once the router's output
  // (ids) is complete; every other mode reads ids / weights before the wait.
  constexpr bool kIdsAfterWait = kMode == kMoeGateUp;

  if (warp == C::kProducerWarp && lane == 0) {
    prefetch_tensormap(&p.tm_w);
    if constexpr (kMode == kMoeGateUp || kMode == kMoeDown) prefetch_tensormap(&p.tm_w2);
    if constexpr (C::kXTma) prefetch_tensormap(&p.tm_x);
  }
  if (tid == 0) {
    s_abort = 0;
    s_last = 0;
    resolve_work<kMode, kT, kNT>(p, s_work, rank);
    for (int i = 0; i < nstages; ++i) {
      mbar_init(smem_u32(&bar_full[i]), C::kFullCount);
      mbar_init(smem_u32(&bar_empty[i]), 1);
    }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(smem_u32(&bar_afull[i]), kT * 128);
      mbar_init(smem_u32(&bar_aempty[i]), 1);
    }
    mbar_init(smem_u32(&bar_accum), 1);
    mbar_init(smem_u32(&bar_inbox), 1);
    mbar_init(smem_u32(&bar_red_ready), S);
    mbar_init(smem_u32(&bar_red_done), S);
    mbar_fence_init();
    if (C::kPush && S > 1) {
      // every rank sends its partials of my rows [r_lo, r_hi) for all tiles
      mbar_arrive_expect_tx(smem_u32(&bar_inbox), S * kT * kNT * (r_hi - r_lo) * 4);
    }
  }
  if (warp == C::kMmaWarp) tmem_alloc(smem_u32(&s_tmem), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (S > 1) {
    if (C::kPush) cluster_arrive();  // paired with a wait before the first remote access
    else cluster_sync();
  }
  // Let the next kernel in the stream start its own prologue (weight
  // prefetch) while this grid runs.  (gate_up routed CTAs have already waited
  // for the router, so a dependent kernel that reads ids early is safe.)
  if (tid == 0) pdl_launch_dependents();

  const CtaWork& wk = s_work;
  const bool active = wk.active != 0;
  const uint32_t tmem = s_tmem;
  const int nst = active ? (wk.k_end - wk.k_begin + C::kStageK - 1) / C::kStageK : 0;

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    const CUtensorMap* tmw = wk.shared ? &p.tm_w2 : &p.tm_w;
    const uint8_t* sfb =
        wk.shared ? p.sf2 : p.sf + (wk.expert >= 0 ? static_cast<size_t>(wk.expert) * p.sf_expert_bytes : 0);
    auto issue_weights = [&](int s) {
      const int slot = s % nstages;
      const uint32_t st = ring + slot * C::kStageBytes;
      const uint32_t fb = smem_u32(&bar_full[slot]);
      const int k0 = wk.k_begin + s * C::kStageK;
      const int kvalid = min(C::kStageK, wk.k_end - k0);
      const int nchunks = kvalid / kSubK;
      uint32_t bytes = kT * C::kWTileBytes;
      if constexpr (C::kFp4) {
        for (int t = 0; t < kT; ++t) bytes += wk.sgroups[t] * nchunks * 512;
      }
      asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(fb), "r"(bytes) : "memory");
      for (int t = 0; t < kT; ++t) {
        const int c0 = C::kFp4 ? k0 / 2 : k0;  // bytes (u8 map) or elements (bf16 map)
        tma_load_2d(st + t * C::kWTileBytes, tmw, c0, wk.wrow[t], fb, pol_w);
        if constexpr (C::kFp4) {
          for (int gi = 0; gi < wk.sgroups[t]; ++gi) {
            const size_t chunk = static_cast<size_t>(wk.srow[t] / 128 + gi) * (wk.kbp / 4) + k0 / 64;
            bulk_load(st + kT * C::kWTileBytes + t * C::kSfTileBytes + gi * 2048, sfb + chunk * 512, nchunks * 512,
                      fb, pol_w);
          }
        }
      }
    };
    const int pre = min(nst, nstages);
    if (lane == 0 && (!kIdsAfterWait || wk.shared)) {
      for (int s = 0; s < pre; ++s) issue_weights(s);
    }
    pdl_wait();
    if (lane == 0 && kIdsAfterWait && !wk.shared) {
      for (int s = 0; s < pre; ++s) issue_weights(s);
    }
    __syncwarp();
    if constexpr (C::kXTma) {
      // Dense activations: rows 0..M-1 of x, one TMA box {64 elements, kNT rows}
      // per 64-wide K atom (rows beyond M read as zeros).
      if (lane == 0) {
        for (int s = 0; s < nst && !s_abort; ++s) {
          const int slot = s % nstages;
          const uint32_t st = ring + slot * C::kStageBytes;
          const uint32_t fb = smem_u32(&bar_full[slot]);
          if (s >= pre) {
            if (!mbar_wait(smem_u32(&bar_empty[slot]), ((s / nstages) & 1) ^ 1, p.err)) { s_abort = 1; break; }
            issue_weights(s);
          }
          const int k0 = wk.k_begin + s * C::kStageK;
          mbar_arrive_expect_tx(fb, C::kXBytes);
          if constexpr (C::kFp4) {
            // one box {64 elements, kNT rows, 4 atoms} of the [K/64, M, 64] view
            tma_load_3d(st + C::kXOff, &p.tm_x, 0, 0, k0 / kSubK, fb, pol_x);
          } else {
            tma_load_2d(st + C::kXOff, &p.tm_x, k0, 0, fb, pol_x);
          }
        }
      }
    } else {
      // Gathered activations (MoE): lane c copies 16-byte chunk c (of 32) of
      // every B row of the stage, 128-byte swizzle.
      const uint16_t* xb = wk.shared ? p.x2 : p.x;
      const int u = lane / 8, cc = lane % 8;
      for (int s = 0; s < nst && !s_abort; ++s) {
        const int slot = s % nstages;
        const uint32_t st = ring + slot * C::kStageBytes;
        const uint32_t fb = smem_u32(&bar_full[slot]);
        if (s >= pre) {
          if (!mbar_wait(smem_u32(&bar_empty[slot]), ((s / nstages) & 1) ^ 1, p.err)) { s_abort = 1; break; }
          if (lane == 0) issue_weights(s);
          __syncwarp();
        }
        const int k0 = wk.k_begin + s * C::kStageK;
        const bool kok = lane * 8 < min(C::kStageK, wk.k_end - k0);
        const uint16_t* src_k = xb + k0 + lane * 8;
        const uint32_t dst0 = st + C::kXOff + u * (kNT * 128);
#pragma unroll 8
        for (int n = 0; n < kNT; ++n) {
          const bool valid = kok && n < wk.ntok;
          const uint32_t dst = dst0 + (n / 8) * 1024 + (n % 8) * 128 + ((cc ^ (n % 8)) * 16);
          cp_async16(dst, valid ? src_k + wk.xoff[n] : xb, valid ? 16u : 0u);
        }
        cp_async_arrive_noinc(fb);
        if (lane == 0) mbar_arrive(fb);
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && active) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kNT);
      int q = 0;
      for (int s = 0; s < nst && !s_abort; ++s) {
        const int slot = s % nstages;
        const uint32_t st = ring + slot * C::kStageBytes;
        const uint32_t xs = st + C::kXOff;
        if constexpr (C::kFp4) {
          const int nsub = min(C::kStageK, wk.k_end - wk.k_begin - s * C::kStageK) / kSubK;
          for (int u = 0; u < nsub; ++u, ++q) {
            const int a = q % kNS;
            if (!mbar_wait(smem_u32(&bar_afull[a]), (q / kNS) & 1, p.err)) { s_abort = 1; break; }
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < kT; ++t) {
              const uint32_t a_tmem = tmem + (a * kT + t) * 32;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t d_tmem = tmem + C::kTmemA + (t * C::kAcc + kk % C::kAcc) * kNT;
                mma_ts(d_tmem, a_tmem + kk * 8, sdesc_sw128(xs + u * (kNT * 128) + kk * 32), idesc,
                       q > 0 || kk >= C::kAcc);
              }
            }
            mma_commit(smem_u32(&bar_aempty[a]));
            if (u == nsub - 1) mma_commit(smem_u32(&bar_empty[slot]));
          }
        } else {
          if (!mbar_wait(smem_u32(&bar_full[slot]), (s / nstages) & 1, p.err)) { s_abort = 1; break; }
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < kT; ++t) {
            const uint32_t ws = st + t * C::kWTileBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t d_tmem = tmem + (t * C::kAcc + kk % C::kAcc) * kNT;
              mma_ss(d_tmem, sdesc_sw128(ws + kk * 32), sdesc_sw128(xs + kk * 32), idesc, s > 0 || kk >= C::kAcc);
            }
          }
          mma_commit(smem_u32(&bar_empty[slot]));
        }
      }
      mma_commit(smem_u32(&bar_accum));
    }
  } else {
    // ------------------------------------------------------------------ dequant warpgroups
    if constexpr (C::kFp4) {
      const int wg = warp / 4;
      const int t = wg % kT;            // tile
      const int g = wg / kT;            // turn: K slices q with q % kG == g
      const int i = tid % 128;          // row in tile
      const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
      const int r = wk.srow[t] + i;     // row in the scale buffer's row space
      const int grp = r / 128 - wk.srow[t] / 128;
      const uint32_t sf_row_off = grp * 2048 + (r % 32) * 16 + ((r % 128) / 32) * 4;
      const uint32_t w_row_off = (i / 8) * 1024 + (i % 8) * 128;
      const uint32_t i8 = i % 8;
      // One K slice: load codes + scales, wait for its tensor-memory slot,
      // permute the activation atom (tile-0 warpgroups), dequantize, store.
      auto slice = [&](uint32_t st, int u, int q) -> bool {
        const uint32_t wt = st + t * C::kWTileBytes + w_row_off;
        const uint4 q0 = lds128(wt + (((2 * u) ^ i8) * 16));
        const uint4 q1 = lds128(wt + (((2 * u + 1) ^ i8) * 16));
        const uint32_t sw = lds32(st + kT * C::kWTileBytes + t * C::kSfTileBytes + sf_row_off + u * 512);
        const int a = q % kNS;
        if (!mbar_wait(smem_u32(&bar_aempty[a]), ((q / kNS) & 1) ^ 1, p.err)) return false;
        tc_fence_after();
        if (t == 0) {
          const uint32_t xa = st + C::kXOff + u * (kNT * 128);
#pragma unroll
          for (int j = i; j < kNT * 8; j += 128) sts128(xa + j * 16, perm_x8(lds128(xa + j * 16)));
        }
        uint32_t s0, s1, s2, s3;
        scale_pair_to_bf16x2(sw & 0xFFFFu, s0, s1);
        scale_pair_to_bf16x2(sw >> 16, s2, s3);
        uint32_t o[16];
        const uint32_t col = tmem + lane_base + (a * kT + t) * 32;
        dequant32_perm(q0, s0, s1, o);
        tmem_st16(col, o);
        dequant32_perm(q1, s2, s3, o);
        tmem_st16(col + 16, o);
        return true;
      };
      int qbase = 0;  // global index of the current stage's first K slice
      for (int s = 0; s < nst && !s_abort; ++s) {
        const int slot = s % nstages;
        const uint32_t st = ring + slot * C::kStageBytes;
        const int nsub = min(C::kStageK, wk.k_end - wk.k_begin - s * C::kStageK) / kSubK;
        const int first = ((g - qbase) % kG + kG) % kG;  // my first slice in this stage
        if (first < nsub) {
          if (!mbar_wait(smem_u32(&bar_full[slot]), (s / nstages) & 1, p.err)) { s_abort = 1; break; }
          // my slices two at a time: one tensor-memory store wait per pair
          for (int u = first; u < nsub; u += 2 * kG) {
            const int u2 = u + kG;
            const bool two = u2 < nsub;
            if (!slice(st, u, qbase + u) || (two && !slice(st, u2, qbase + u2))) { s_abort = 1; break; }
            tmem_wait_st();
            if (t == 0) fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_afull[(qbase + u) % kNS]));
            if (two) mbar_arrive(smem_u32(&bar_afull[(qbase + u2) % kNS]));
          }
        }
        qbase += nsub;
      }
    }
  }

  // ==================================================================== epilogue
  __syncwarp();
  if (warp < 4 * C::kWarpgroups) {
    const int wg = warp / 4;  // warpgroups 0 .. kT-1 read tile wg's accumulator
    const int i = tid % 128;
    const bool ok_acc = active && mbar_wait(smem_u32(&bar_accum), 0, p.err);
    if (!ok_acc && active) s_abort = 1;
    tc_fence_after();
    const float post = C::kFp4 ? static_cast<float>(1 << kShift) : 1.0f;
    // Partials of (tile t, token n, row i).  Push mode: rank `rank` owns rows
    // [r_lo, r_hi) and receives them from every rank into
    // inbox[src][t][n][row - r_lo]; pull mode: each rank leaves its partials in
    // its own ring as red[t][n][row] and the owner reads them through DSMEM.
    if constexpr (C::kPush) {
      if (S > 1) cluster_wait();  // all peers' inbox barriers are initialised
      if (active && wg < kT) {
        const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
        const uint32_t dcol = tmem + lane_base + C::kTmemA + wg * C::kAcc * kNT;
        const uint32_t owner = static_cast<uint32_t>(i / R);
        const int rr = i - static_cast<int>(owner) * R;
        const int rows_owner = min(R, 128 - static_cast<int>(owner) * R);
        const uint32_t base = inbox + ((rank * kT + wg) * kNT * rows_owner + rr) * 4;
        const uint32_t rbase = S > 1 ? mapa(base, owner) : base;
        const uint32_t rbar = S > 1 ? mapa(smem_u32(&bar_inbox), owner) : 0u;
#pragma unroll
        for (int c = 0; c < kNT; c += 8) {
          float acc8[8];
          load_acc<C::kAcc, kNT>(dcol + c, acc8);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float val = acc8[j] * post;
            const uint32_t off = (c + j) * rows_owner * 4;
            if (S > 1) st_async_f32(rbase + off, val, rbar);
            else stsf(rbase + off, val);
          }
        }
      }
      tc_fence_before();
      if (S > 1) {
        if (!mbar_wait<true>(smem_u32(&bar_inbox), 0, p.err)) s_abort = 1;
      } else {
        epi_sync<kEpiThreads>();
      }
    } else {
      epi_sync<kEpiThreads>();  // every ring stage is consumed: reuse it for partials
      if (active && !s_abort && wg < kT) {
        const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
        const uint32_t dcol = tmem + lane_base + C::kTmemA + wg * C::kAcc * kNT;
#pragma unroll
        for (int c = 0; c < kNT; c += 8) {
          float acc8[8];
          load_acc<C::kAcc, kNT>(dcol + c, acc8);
#pragma unroll
          for (int j = 0; j < 8; ++j) stsf(ring + ((wg * kNT + c + j) * 128 + i) * 4, acc8[j] * post);
        }
      }
      tc_fence_before();
      epi_sync<kEpiThreads>();
      if (S > 1) {
        if (tid == 0) {
          for (uint32_t r2 = 0; r2 < S; ++r2) mbar_arrive_cluster(mapa(smem_u32(&bar_red_ready), r2));
        }
        if (!mbar_wait<true>(smem_u32(&bar_red_ready), 0, p.err)) s_abort = 1;
      }
    }
    // Sum over the cluster ranks, in rank order, of the partial of
    // (tile t, token n, row) for a row this rank owns.
    auto partial = [&](int t, int n, int row) -> float {
      if constexpr (C::kPush) {
        const int rows_mine = r_hi - r_lo;
        float acc = 0.0f;
        for (uint32_t src = 0; src < S; ++src)
          acc += ldsf(inbox + (((src * kT + t) * kNT + n) * rows_mine + (row - r_lo)) * 4);
        return acc;
      } else {
        const uint32_t off = ring + ((t * kNT + n) * 128 + row) * 4;
        if (S == 1) return ldsf(off);
        float acc = 0.0f;
        for (uint32_t r2 = 0; r2 < S; ++r2) {
          float v;
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(mapa(off, r2)) : "memory");
          acc += v;
        }
        return acc;
      }
    };
    if (active && !s_abort) {
      pdl_wait();
      if constexpr (kMode == kDenseFp4 || kMode == kDenseBf16) {
        const float gs = p.gs ? __ldg(p.gs) : 1.0f;
        for (int it = tid; it < (r_hi - r_lo) * wk.ntok; it += kEpiThreads) {
          const int n = it / (r_hi - r_lo), row = r_lo + it % (r_hi - r_lo);
          const int o = wk.out_base + row;
          if (o >= p.n_out) continue;
          uint16_t res;
          if (kT == 1) {
            res = f32_to_bf16_rn(partial(0, n, row) * gs);
          } else {
            const float G = bf16_to_f32(f32_to_bf16_rn(partial(0, n, row) * gs));
            const float U = bf16_to_f32(f32_to_bf16_rn(partial(1, n, row) * gs));
            res = f32_to_bf16_rn(silu_exact(G) * U);
          }
          p.out[static_cast<int64_t>(n) * p.ldo + o] = res;
        }
      } else if constexpr (kMode == kMoeGateUp) {
        if (!wk.shared) {
          const float al = __ldg(p.alpha + wk.expert);
          for (int it = tid; it < kT * 64 * wk.ntok; it += kEpiThreads) {
            const int n = it / (kT * 64), rem = it % (kT * 64);
            const int t = rem / 64, o = rem % 64;
            const int feat = blockIdx.x * (kT * 64) + t * 64 + o;
            if (feat >= p.n_out) continue;
            const float u = partial(t, n, o) * al;
            const float gt = partial(t, n, o + 64) * al;
            p.out[static_cast<int64_t>(wk.orow[n]) * p.ldo + feat] = f32_to_bf16_rn(silu_fast(gt) * u);
          }
        } else {
          const float gs = __ldg(p.gs);
          for (int it = tid; it < 128 * wk.ntok; it += kEpiThreads) {
            const int n = it / 128, row = it % 128;
            const int o = wk.out_base + row;
            if (o >= p.shared_n_out) continue;
            const float G = bf16_to_f32(f32_to_bf16_rn(partial(0, n, row) * gs));
            const float U = bf16_to_f32(f32_to_bf16_rn(partial(1, n, row) * gs));
            p.out2[static_cast<int64_t>(wk.orow[n]) * p.ldo2 + o] = f32_to_bf16_rn(silu_exact(G) * U);
          }
        }
      } else {  // kMoeDown: y values into the scratch
        const float sc = wk.shared ? __ldg(p.gs) : __ldg(p.alpha + wk.expert);
        uint16_t* dst = wk.shared ? p.out2 : p.out;
        const int64_t ld = wk.shared ? p.ldo2 : p.ldo;
        const int nfeat = wk.shared ? p.shared_n_out : p.n_out;
        for (int it = tid; it < 128 * wk.ntok; it += kEpiThreads) {
          const int n = it / 128, row = it % 128;
          const int o = wk.out_base + row;
          if (o >= nfeat) continue;
          dst[static_cast<int64_t>(wk.orow[n]) * ld + o] = f32_to_bf16_rn(partial(0, n, row) * sc);
        }
      }
    }
    if (!C::kPush && S > 1) {
      epi_sync<kEpiThreads>();
      if (tid == 0) {
        for (uint32_t r2 = 0; r2 < S; ++r2) mbar_arrive_cluster(mapa(smem_u32(&bar_red_done), r2));
      }
      if (!mbar_wait<true>(smem_u32(&bar_red_done), 0, p.err)) s_abort = 1;
    }
    if constexpr (kMode == kMoeDown) {
      // Every CTA of a row-tile column arrives once; the last one combines.
      epi_sync<kEpiThreads>();
      if (tid == 0) {
        // Arrival count tagged with this call's epoch: a counter holding any
        // other epoch (an earlier call, or never-initialised scratch) counts
        // as zero, so the workspace needs no zero-fill.  The last arrival
        // resets the counter.
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
        const int h0 = blockIdx.x * 128;
        for (int it = tid; it < 128 * p.M; it += kEpiThreads) {
          const int t = it / 128, h = h0 + it % 128;
          if (h >= p.n_out) continue;
          bool ids_ok = true;  // a token with an out-of-range id is left unwritten
          for (int j = 0; j < p.topk; ++j) {
            const int e = __ldg(p.ids + t * p.topk + j);
            ids_ok = ids_ok && e >= 0 && e < p.E;
          }
          if (!ids_ok) continue;
          float acc = 0.0f;
          for (int j = 0; j < p.topk; ++j) {
            const float wj = __ldg(p.tw + t * p.topk + j);
            const float y = bf16_to_f32(__ldcg(p.out + static_cast<int64_t>(t * p.topk + j) * p.ldo + h));
            acc = fmaf(wj, y, acc);
          }
          const float sb = bf16_to_f32(f32_to_bf16_rn(acc));
          const float ysh = bf16_to_f32(__ldcg(p.out2 + static_cast<int64_t>(t) * p.ldo2 + h));
          p.out3[static_cast<int64_t>(t) * p.n_out + h] = f32_to_bf16_rn(sb + ysh);
        }
      }
    }
  } else if (C::kPush && S > 1) {
    cluster_wait();  // the producer and MMA warps close their cluster-barrier phase
  }

  // ==================================================================== teardown
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fp4
