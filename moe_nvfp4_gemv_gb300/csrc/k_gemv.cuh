// k_gemv.cuh -- the small-M GEMV pipeline on tcgen05 tensor cores.
//
// One kernel template serves the dense NVFP4 GEMV above 16 tokens
// (optionally with the fused silu_mul epilogue), the BF16-weight GEMV, and
// both MoE kernels above 64 tokens (vllm.models.flint.ops.nvfp4_gemv
// nvfp4_gemv / bf16_gemv, vllm.models.flint.ops.moe_gemv gate_up /
// down_combine).
//
// Swap-AB: a CTA owns one tile of 128 weight rows (the MMA M dimension); the
// tokens are the MMA N dimension (kNT = 16 .. 128).  A tile is either 128
// consecutive rows or, for the silu_mul epilogue, two 64-row boxes: 64 gate
// rows and the 64 up rows of the same output features, so one CTA holds both
// operands of its outputs.  Its K range is a slice of K; the S CTAs of a
// cluster split K and reduce their fp32 partials through distributed shared
// memory in rank order (deterministic).
//
// Warp roles (kW dequant warpgroups, then a weight producer warp, an MMA
// warp and, NVFP4 only, an activation producer warp and, for tiles of up to
// 32 tokens, a permute warp):
//   weights   lane 0 streams weight boxes (TMA, 128-byte swizzle) and the
//             matching 512-byte scale chunks (bulk copies) into a ring of
//             shared-memory stages of 256 K; with PDL the first stages are
//             issued before griddepcontrol.wait.  A stage is refilled once
//             the dequant warps have read the stage that held its slot.
//   activations  (NVFP4) after the wait, into a ring of their own, one 128-K
//             slice per slot (TMA for dense rows, cp.async gathers by all 32
//             lanes for MoE), refilled once the slice's MMAs are done, so
//             the weight ring, which hides HBM latency, is not shortened by
//             activations that come from L2.  BF16: a stage's activations
//             travel in the weight stage, loaded by the weight producer.
//   permute   (NVFP4, up to 32 tokens) as each slice lands, its activations
//             in place into the weight pairs' K order (dequant.cuh), then an
//             arrival the MMA warp waits for, so the dequant warps never wait
//             for activations (measured at 32 tokens: ~0.6 us of waiting and
//             ~0.3 us of permuting per slice when they did).  Larger tiles:
//             the dequant warps permute their share of each slice (one warp
//             was too slow for 64 and 128 tokens).
//   dequant   warpgroup w takes the 128-wide K slices q = w, w + kW, ...  For
//             each slice thread i (row i) reads its code bytes and scale
//             bytes (then frees its warp's share of the weight stage),
//             dequantizes them exactly to bf16 (dequant.cuh) and stores them
//             with tcgen05.st into the slice's tensor-memory A slot (a ring
//             of kSlots slots shared by the warpgroups), then arrive on the
//             slot's barrier.
//   MMA       the warp waits for each slot (and its permuted activation
//             slice) together and one elected lane
//             issues the slot's eight K=16 tcgen05.mma into the fp32
//             accumulator and frees the tensor-memory slot and the slice's
//             activation slot with tcgen05.commit, so the dequant warps never
//             wait on MMA issue.
//   epilogue  the dequant warps read the accumulator (tcgen05.ld), exchange
//             partials through (distributed) shared memory and apply the
//             mode's epilogue.
// The BF16-weight mode has no dequant step: the MMA warp issues tcgen05.mma
// with both operands in shared memory, and one warpgroup runs the epilogue.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "dequant.cuh"

namespace fp4 {

enum Mode : int {
  kDenseFp4 = 0,   // nvfp4_gemv, optionally with silu_mul ([gate | up] halves)
  kDenseBf16 = 1,  // bf16_gemv and the GEMM of the dequantize + GEMM path
  kMoeGateUp = 2,  // routed experts ([up; gate] 64-row groups) + shared expert
  kMoeDown = 3,    // routed + shared experts into scratch, last CTA combines
};

constexpr int kMaxStages = 8;
constexpr int kSubK = 64;       // K per A slot / per activation atom
constexpr int kStageK4 = 256;   // K per ring stage, NVFP4 weights (128 B per row)
constexpr int kStageK16 = 64;   // K per ring stage, bf16 weights (128 B per row)
constexpr int kMaxNT = 128;
constexpr int kMaxWG = 2;
constexpr int kMaxSlots = 6;
constexpr int kMaxXSlots = 4;   // activation slots (NVFP4 modes; the host picks 2, 3 or 4)
constexpr int kSliceK = 128;    // K per tensor-memory A slot (8 MMAs of K = 16 per commit)
constexpr int kSlabMaxStages = 64;  // slab kernel: K per CTA <= 64 stages of 256
constexpr int kSlabMaxCW = 4;       // slab kernel: consumer warps (tiles of 16 kSlabR cw rows: 64 or 128)
constexpr int kSlabChunk = 4;       // slab kernel, MoE: pairs of one expert per CTA (B rows)
constexpr int kSlabNT = 8;          // slab kernel: MMA N (tokens / pairs 0 .. 7)
constexpr int SlabInboxBytes = 8 * (128 + 16) * 4;  // slab kernel: split-K inbox (8 tokens x 144 rows, fp32)

struct GemvParams {
  CUtensorMap tm_w;    // weights read by routed / dense CTAs
  CUtensorMap tm_w2;   // shared-expert weights (MoE)
  CUtensorMap tm_x;    // dense modes: activations (TMA)
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
  int n_half;          // paired tiles: first up row (dense silu: N / 2; shared gate_up: SI)
  int silu;            // dense: 1 = silu_mul epilogue (paired tiles)
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
  int nstages;         // weight ring stages
  int nx;              // tcgen05 NVFP4 modes: activation slots (one 128-K slice each)
  int wstage;          // tcgen05 NVFP4 modes: bytes per weight stage (codes + sf_slots scale groups)
  int sf_slots;        // tcgen05 NVFP4 modes: 2 KB scale-group slots per weight stage (1 .. 3)
  int inbox_off;       // tcgen05 push mode: offset of the split-K inbox from the ring (0: the drained ring)
  int stage_bytes;     // register-fed kernel: bytes per ring stage (weights, scale groups, activations);
                       // slab kernel: bytes per ring stage (weights, scale groups)
  int x_off;           // register-fed kernel: offset of the activations in a stage; slab kernel:
                       // bytes of the activation slab (the ring starts there)
  int cw;              // register-fed dense kernel: consumer warps = tile height / 16 (4 .. 8);
                       // slab kernel: consumer warps (2 or 4), tile height 16 slab_r cw
  int slab_r;          // slab kernel: 16-row blocks per consumer warp (1 or 2)
  int tiles_per_cta;   // slab kernel, down_combine: 128-row tiles one CTA streams in turn
  int chunk;           // MoE: pairs (shared expert: tokens) per CTA column chunk, 1 .. kNT (0: kNT)
  int skip_stage;      // test hook: the dense producers issue nothing for this 256-K stage (-1: none)
  uint32_t* err;       // device error word (the wait limit follows it, see common.cuh)
};

// kN: the most B rows a CTA holds (the token tile, or the slab kernel's
// expert chunk).
template <int kN>
struct CtaWorkN {
  int active;      // 0: nothing to compute
  int shared;      // 1: shared-expert CTA (MoE)
  int paired;      // 1: two 64-row boxes (gate rows, up rows); 0: one 128-row box
  int ntok;        // valid B rows
  int k_begin, k_end;
  int wrow[2];     // tensor-map row of each box
  int srow[2];     // scale-buffer row of each box's first row
  int sgroup[3];   // 128-row scale groups copied per stage: box 0's, then box 1's first and
                   // second (a 64-row box that starts off a 64-row boundary straddles two);
                   // -1: none (beyond the buffer, or not needed)
  int kbp;
  int expert;
  int out_base;    // first output feature of the tile
  int tok[kN];   // B row -> activation row
  int orow[kN];  // B row -> output row (pair / token)
  long long xoff[kN];  // B row -> element offset of its activation row
};
using CtaWork = CtaWorkN<kMaxNT>;

__host__ __device__ constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p *= 2;
  return p;
}

template <int kMode, int kNT>
struct Cfg {
  static constexpr bool kFp4 = kMode != kDenseBf16;
  static constexpr int kW = kFp4 ? 2 : 1;  // worker warpgroups
  // NVFP4: a third warp streams the activation ring; up to 32 tokens a
  // fourth permutes each landed activation slice for the MMAs (larger tiles:
  // the dequant warps permute it, a slice being too much for one warp)
  static constexpr bool kPermSep = kFp4 && kNT <= 32;
  static constexpr int kThreads = kW * 128 + (kFp4 ? (kPermSep ? 128 : 96) : 64);
  static constexpr int kProducerWarp = 4 * kW;
  static constexpr int kMmaWarp = 4 * kW + 1;
  static constexpr int kXWarp = 4 * kW + 2;
  static constexpr int kPermWarp = kPermSep ? 4 * kW + 3 : -1;
  static constexpr int kStageK = kFp4 ? kStageK4 : kStageK16;
  static constexpr int kSlicesPerStage = kFp4 ? kStageK / kSliceK : 1;  // 2 (fp4) or 1 (bf16)
  static constexpr int kWTileBytes = 128 * 128;
  static constexpr int kSfTileBytes = kFp4 ? 3 * 4 * 512 : 0;  // three 128-row scale groups x 4 chunks
  static constexpr int kXBytes = kNT * kStageK * 2;
  static constexpr int kXOff = kWTileBytes + kSfTileBytes;
  static constexpr int kStageBytes = kXOff + kXBytes;  // BF16: weights and activations of a stage
  // NVFP4: activations have a ring of their own, one 128-K slice per slot
  // (two 64-K atoms of kNT rows x 128 bytes).
  static constexpr int kXSliceBytes = kNT * kSliceK * 2;
  // Tensor memory: one fp32 accumulator (kNT columns), then a ring of kSlots
  // A slots (64 columns = 128 bf16 K each) shared by the warpgroups in slice
  // order.  256 columns (two CTAs per SM) up to kNT = 64.
  static constexpr int kAccCols = kNT;
  static constexpr int kSlotCols = kSliceK / 2;
  static constexpr int kSlots = !kFp4 ? 0 : kNT <= 64 ? 3 : 6;
  static constexpr int kTmemCols = pow2_at_least(kAccCols + kSlots * kSlotCols);
  static constexpr int kRedBytes = kNT * 128 * 4;
  // Dense modes read contiguous activation rows with TMA; the MoE modes
  // gather rows by token / pair with cp.async from the producer lanes.
  static constexpr bool kXTma = kMode == kDenseFp4 || kMode == kDenseBf16;
  static constexpr int kFullCount = kXTma ? 1 : 33;
  // Split-K partials are pushed to the owning cluster rank (st.async into a
  // dedicated inbox) when the inbox is small; otherwise pulled through DSMEM
  // from the (reused) ring.
  static constexpr bool kPush = kNT <= 32;
  static constexpr int kInboxBytes = kPush ? kNT * 136 * 4 : 0;
  static_assert(kNT % 16 == 0 && kNT >= 16 && kNT <= kMaxNT, "token tile");
  static_assert(kStageBytes % 1024 == 0 && kXSliceBytes % 1024 == 0, "stage alignment");
  static_assert(kTmemCols <= 512, "tensor memory");
  static_assert(kSlots <= kMaxSlots && kW <= kMaxWG, "barrier arrays");
  // CTAs per SM the launch aims for (tensor memory is 512 columns per SM)
  static constexpr int kMinBlocks = kTmemCols <= 256 ? 2 : 1;
};

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// down_combine of 8 consecutive h of token t: out[t, h .. h + 7] =
// bf16(bf16(sum_j tw[t, j] * y[t, j, h]) + y_shared[t, h]), the sum in fp32
// over j = 0 .. topk - 1 with fused multiply-adds (16-byte loads of y and
// y_shared, one 16-byte store).  The loads of up to kJ j are issued before
// any is used (one round trip per group of kJ, not per j); the sum keeps the
// j order, so kJ does not change the result.  A token with an out-of-range
// id is left unwritten.
template <int kJ = 8>
__device__ __forceinline__ void moe_combine_item(const GemvParams& p, int t, int h) {
  const uint4 sv = __ldcg(reinterpret_cast<const uint4*>(p.out2 + static_cast<int64_t>(t) * p.ldo2 + h));
  bool ids_ok = true;
  float a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = 0.0f;
  for (int j0 = 0; j0 < p.topk; j0 += kJ) {
    int e[kJ];
    float wj[kJ];
    uint4 yv[kJ];
#pragma unroll
    for (int jj = 0; jj < kJ; ++jj) {
      const int j = j0 + jj;
      e[jj] = 0;
      wj[jj] = 0.0f;
      yv[jj] = make_uint4(0u, 0u, 0u, 0u);
      if (j < p.topk) {
        e[jj] = __ldg(p.ids + t * p.topk + j);
        wj[jj] = __ldg(p.tw + t * p.topk + j);
        yv[jj] = __ldcg(reinterpret_cast<const uint4*>(p.out + static_cast<int64_t>(t * p.topk + j) * p.ldo + h));
      }
    }
#pragma unroll
    for (int jj = 0; jj < kJ; ++jj) {
      if (j0 + jj >= p.topk) break;
      ids_ok = ids_ok && e[jj] >= 0 && e[jj] < p.E;
      const uint32_t yw[4] = {yv[jj].x, yv[jj].y, yv[jj].z, yv[jj].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[2 * q] = fmaf(wj[jj], __uint_as_float(yw[q] << 16), a[2 * q]);
        a[2 * q + 1] = fmaf(wj[jj], __uint_as_float(yw[q] & 0xFFFF0000u), a[2 * q + 1]);
      }
    }
  }
  if (!ids_ok) return;
  const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float lo = __uint_as_float(static_cast<uint32_t>(f32_to_bf16_rn(a[2 * q])) << 16) +
                     __uint_as_float(sw[q] << 16);
    const float hi = __uint_as_float(static_cast<uint32_t>(f32_to_bf16_rn(a[2 * q + 1])) << 16) +
                     __uint_as_float(sw[q] & 0xFFFF0000u);
    o[q] = static_cast<uint32_t>(f32_to_bf16_rn(lo)) | (static_cast<uint32_t>(f32_to_bf16_rn(hi)) << 16);
  }
  *reinterpret_cast<uint4*>(p.out3 + static_cast<int64_t>(t) * p.n_out + h) = make_uint4(o[0], o[1], o[2], o[3]);
}

// down_combine of one 128-row tile of H (rows h0 .. h0 + 127) by `nthr`
// threads (this one is `ti`); a work item is 8 consecutive h of one token
// (H is a multiple of 64, so an item is wholly inside or outside H).
template <int kJ = 8>
__device__ __forceinline__ void moe_combine_tile(const GemvParams& p, int h0, int ti, int nthr) {
  for (int it = ti; it < 16 * p.M; it += nthr) {
    const int t = it / 16, h = h0 + 8 * (it % 16);
    if (h < p.n_out) moe_combine_item<kJ>(p, t, h);
  }
}

// Tag a down_combine CTA leaves in a tile's counter when it gave up (a wait
// ran out): the slab kernel's calls combine in a kernel of their own, which
// skips tiles tagged with its call's epoch, so their outputs stay unwritten.
__host__ __device__ constexpr unsigned long long abort_tag(uint32_t epoch) {
  return (static_cast<unsigned long long>(epoch) << 32) | 0xFFFFFFFFull;
}

// SiLU with IEEE exp and division (the "exact" SiLU of the dense path).
__device__ __forceinline__ float silu_exact(float g) { return __fdiv_rn(g, 1.0f + expf(-g)); }
// SiLU with the fast exponential and division (the routed experts' fast sigmoid).
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Named barriers: 1 = all worker threads; 2 + w = warpgroup w.
template <int kThreadsEpi>
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreadsEpi) : "memory");
}

// Rows of a tile are reduced across cluster ranks per feature unit: a tile
// whose feature o combines rows o and o + 64 (paired gate/up boxes, routed
// [up; gate] groups) has 64-row units, any other tile 128-row units.
template <int kMode>
__device__ __forceinline__ int feature_unit(const CtaWork& w) {
  return (w.paired || (kMode == kMoeGateUp && !w.shared)) ? 64 : 128;
}

// Tensor-map row, scale row and scale groups of one box (box 0: 128 or 64
// rows starting on a group or half-group boundary, one group; box 1: 64 rows,
// one or two groups).
template <typename Work>
__device__ __forceinline__ void set_box(Work& w, int b, int wrow, int srow, int groups_total) {
  w.wrow[b] = wrow;
  w.srow[b] = srow;
  const int g0 = srow / 128;
  if (b == 0) {
    w.sgroup[0] = g0 < groups_total ? g0 : -1;
  } else {
    const int g1 = (srow + 63) / 128;
    w.sgroup[1] = g0 < groups_total ? g0 : -1;
    w.sgroup[2] = (g1 != g0 && g1 < groups_total) ? g1 : -1;
  }
}

// Resolve what a CTA computes for row tile (or tile group) `tile` of grid
// column `col` (called by all 32 lanes of the producer warp).  gate_up
// routed CTAs wait for the previous grid first: their expert ids come from
// the router.  A routed CTA's chunk is found with warp-wide ballots over the
// ids, so resolving costs O(P / 32) loads per lane however many pairs there
// are.
template <int kMode, int kNT, typename Work = CtaWork>
__device__ void resolve_work_at(const GemvParams& p, Work& w, uint32_t split, int lane, int tile, int col) {
  // pairs (tokens) per MoE chunk: p.chunk when the host set one (1 .. kNT), else kNT
  const int cn = p.chunk > 0 && p.chunk < kNT ? p.chunk : kNT;
  if (lane == 0) {
    w.active = 1;
    w.shared = 0;
    w.paired = 0;
    w.expert = -1;
    w.sgroup[1] = w.sgroup[2] = -1;
    w.wrow[1] = w.srow[1] = 0;
  }
  if constexpr (kMode == kDenseFp4 || kMode == kDenseBf16) {
    if (lane == 0) {
      w.ntok = p.M;  // B row n is token n (activations read by TMA)
      w.k_begin = static_cast<int>(split) * p.k_split;
      w.k_end = min(p.K, w.k_begin + p.k_split);
      w.kbp = p.kbp;
      const int groups_total = (p.rows_w + 127) / 128;
      if (p.silu) {
        w.paired = 1;
        w.out_base = tile * 64;
        set_box(w, 0, tile * 64, tile * 64, groups_total);                        // gate rows
        set_box(w, 1, p.n_half + tile * 64, p.n_half + tile * 64, groups_total);  // up rows
      } else {
        w.out_base = tile * 128;
        set_box(w, 0, tile * 128, tile * 128, groups_total);
      }
    }
  } else {
    // MoE: blockIdx.y < P: routed pair column; else shared-expert token chunk.
    if (lane == 0) w.k_begin = 0;
    if (col < p.P) {
      // gate_up runs right after the router: its ids are complete only after
      // the wait.  down_combine reads them early (they are two kernels old).
      if (kMode == kMoeGateUp) pdl_wait();
      // ids of pairs 0 .. 63 (lane, lane + 32) load together with this
      // column's, so resolving costs one global round trip for up to 64 pairs
      const int id0 = lane < p.P ? __ldg(p.ids + lane) : -1;
      const int id1 = lane + 32 < p.P ? __ldg(p.ids + lane + 32) : -1;
      const int e = __ldg(p.ids + col);
      bool live = tile < p.routed_tiles;
      if (live && (e < 0 || e >= p.E)) {
        if (lane == 0) raise_error(p.err, FP4_ERR_BADIDX);
        live = false;
      }
      // rank of this pair among the pairs routed to e; the first pair of each
      // chunk of `cn` pairs computes the whole chunk.
      int cnt = 0;
      if (live)
        for (int q = lane; q < col; q += 32) cnt += ((q < 32 ? id0 : q < 64 ? id1 : __ldg(p.ids + q)) == e);
      const int rank = __reduce_add_sync(0xFFFFFFFFu, cnt);
      live = live && rank % cn == 0;
      if (!live) {
        if (lane == 0) w.active = 0;
        __syncwarp();
        return;
      }
      // the chunk: the first cn pairs q >= col routed to e, in order
      int n = 0;
      for (int q0 = col; q0 < p.P && n < cn; q0 += 32) {
        const int q = q0 + lane;
        const int v0 = __shfl_sync(0xFFFFFFFFu, id0, q % 32);
        const int v1 = __shfl_sync(0xFFFFFFFFu, id1, q % 32);
        const int idq = q < 32 ? v0 : q < 64 ? v1 : (q < p.P ? __ldg(p.ids + q) : -1);
        const bool m = q < p.P && idq == e;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, m);
        const int pos = n + __popc(bal & ((1u << lane) - 1u));
        if (m && pos < cn) {
          w.tok[pos] = kMode == kMoeGateUp ? q / p.topk : q;  // x row (token) or act row (pair)
          w.orow[pos] = q;
        }
        n += __popc(bal);
      }
      n = min(n, cn);
      __syncwarp();
      if (lane == 0) {
        w.ntok = n;
        for (int i = n; i < kNT; ++i) w.tok[i] = w.orow[i] = w.tok[0];
        w.expert = e;
        w.k_end = p.K;
        w.kbp = p.kbp;
        // 128 consecutive rows of expert e (gate_up: one [up; gate] group)
        const int r0 = tile * 128;
        set_box(w, 0, e * p.rows_per_expert + r0, r0, (p.rows_per_expert + 127) / 128);
        w.out_base = kMode == kMoeGateUp ? tile * 64 : tile * 128;
      }
      __syncwarp();
      for (int m2 = lane; m2 < kNT; m2 += 32) w.xoff[m2] = static_cast<long long>(w.tok[m2]) * p.ldx;
    } else if (lane == 0) {
      const int chunk = col - p.P;
      if (tile >= p.shared_tiles) {
        w.active = 0;
      } else {
        w.shared = 1;
        const int t0 = chunk * cn;
        w.ntok = min(cn, p.M - t0);
        for (int n = 0; n < kNT; ++n) w.tok[n] = w.orow[n] = t0 + (n < w.ntok ? n : 0);
        w.k_end = p.K2;
        w.kbp = p.kbp2;
        const int groups_total = (p.rows_w + 127) / 128;
        if (kMode == kMoeGateUp) {
          w.paired = 1;
          w.out_base = tile * 64;
          set_box(w, 0, tile * 64, tile * 64, groups_total);                        // gate rows
          set_box(w, 1, p.n_half + tile * 64, p.n_half + tile * 64, groups_total);  // up rows
        } else {
          w.out_base = tile * 128;
          set_box(w, 0, tile * 128, tile * 128, groups_total);
        }
        for (int m = 0; m < kNT; ++m) w.xoff[m] = static_cast<long long>(w.tok[m]) * p.ldx2;
      }
    }
  }
  __syncwarp();
}

// The work of this CTA of the grid (tile from blockIdx.x over the cluster,
// column blockIdx.y), before the barriers are initialised.
template <int kMode, int kNT, typename Work = CtaWork>
__device__ void resolve_work(const GemvParams& p, Work& w, uint32_t split, int lane) {
  resolve_work_at<kMode, kNT, Work>(p, w, split, lane, static_cast<int>(blockIdx.x / max(1u, cluster_nctarank())),
                                    static_cast<int>(blockIdx.y));
}

template <int kMode, int kNT>
__global__ void __launch_bounds__(Cfg<kMode, kNT>::kThreads, Cfg<kMode, kNT>::kMinBlocks)
    gemv_kernel(const __grid_constant__ GemvParams p) {
  using C = Cfg<kMode, kNT>;
  constexpr int kW = C::kW;
  constexpr int kEpiThreads = kW * 128;
  constexpr int kNS = C::kSlots;
  constexpr int kSPS = C::kSlicesPerStage;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-aligned ring, addressed through 32-bit shared-window addresses:
  // the weight stages, then (NVFP4) the activation slots; the split-K inbox
  // (push mode) follows, or with one rank reuses the drained ring.
  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int wstage = C::kFp4 ? p.wstage : C::kStageBytes;
  const uint32_t xring = ring + p.nstages * wstage;
  const int nx = p.nx;
  const uint32_t inbox = ring + p.inbox_off;
  __shared__ __align__(8) uint64_t bar_full[kMaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kMaxStages];   // NVFP4: stage dequantized; BF16: its MMAs done
  __shared__ __align__(8) uint64_t bar_xfull[kMaxXSlots];   // activation slice landed
  __shared__ __align__(8) uint64_t bar_xempty[kMaxXSlots];  // activation slice's MMAs done (MMA-thread commit)
  __shared__ __align__(8) uint64_t bar_xready[kMaxXSlots];  // activation slice permuted (permute warp)
  __shared__ __align__(8) uint64_t bar_afull[kMaxSlots];   // slot dequantized (4 warps of its warpgroup)
  __shared__ __align__(8) uint64_t bar_aempty[kMaxSlots];  // slot's MMAs done (MMA-thread commit)
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

  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_x = policy_evict_last();

  // ------------------------------------------------------------------ prologue
  // The producer resolves the work (gate_up routed CTAs: after the wait for
  // the router's ids) and initialises every barrier before the CTA-wide
  // barrier; warp 0 allocates tensor memory meanwhile.  The weight stream
  // starts right after it.
  int pre = 0;  // stages whose weights the producer has issued
  auto stage_count = [&](const CtaWork& wk) {
    return wk.active ? (wk.k_end - wk.k_begin + C::kStageK - 1) / C::kStageK : 0;
  };
  // Weights of stage s into its ring slot.  NVFP4: the stage's full barrier
  // counts this arrival and the code and scale bytes; BF16: only the bytes
  // (the activations' load arrives).  A stage holds p.sf_slots scale groups;
  // a group beyond them (which the host's sizing rules out) is reported and
  // not copied.
  auto issue_weights = [&](const CtaWork& wk, int s) {
    const int slot = s % nstages;
    const uint32_t st = ring + slot * wstage;
    const uint32_t fb = smem_u32(&bar_full[slot]);
    const int k0 = wk.k_begin + s * C::kStageK;
    const int kvalid = min(C::kStageK, wk.k_end - k0);
    const int nchunks = kvalid / kSubK;
    const CUtensorMap* tmw = wk.shared ? &p.tm_w2 : &p.tm_w;
    uint32_t bytes = C::kWTileBytes;
    if constexpr (C::kFp4) {
      for (int g = 0; g < 3; ++g) {
        if (wk.sgroup[g] < 0) continue;
        if (g >= p.sf_slots) {
          raise_error(p.err, FP4_ERR_BADIDX);
          continue;
        }
        bytes += nchunks * 512;
      }
      mbar_arrive_expect_tx(fb, bytes);
    } else {
      asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(fb), "r"(bytes) : "memory");
    }
    const int c0 = C::kFp4 ? k0 / 2 : k0;  // bytes (u8 map) or elements (bf16 map)
    tma_load_2d(st, tmw, c0, wk.wrow[0], fb, pol_w);
    if (wk.paired) tma_load_2d(st + C::kWTileBytes / 2, tmw, c0, wk.wrow[1], fb, pol_w);
    if constexpr (C::kFp4) {
      const uint8_t* sfb =
          wk.shared ? p.sf2 : p.sf + (wk.expert >= 0 ? static_cast<size_t>(wk.expert) * p.sf_expert_bytes : 0);
      for (int g = 0; g < 3 && g < p.sf_slots; ++g) {
        if (wk.sgroup[g] < 0) continue;
        const size_t chunk = static_cast<size_t>(wk.sgroup[g]) * (wk.kbp / 4) + k0 / 64;
        bulk_load(st + C::kWTileBytes + g * 2048, sfb + chunk * 512, nchunks * 512, fb, pol_w);
      }
    }
  };

  if (warp == C::kProducerWarp) resolve_work<kMode, kNT>(p, s_work, rank, lane);
  if (warp == C::kProducerWarp && lane == 0) {
    prefetch_tensormap(&p.tm_w);
    if constexpr (kMode == kMoeGateUp || kMode == kMoeDown) prefetch_tensormap(&p.tm_w2);
    if constexpr (C::kXTma) prefetch_tensormap(&p.tm_x);
    s_abort = 0;
    s_last = 0;
    CtaWork& wk = s_work;
    const int nst = stage_count(wk);
    for (int i = 0; i < nstages; ++i) {
      // NVFP4: the weights' arrival; a stage is free once every warp of the
      // warpgroups that dequantize its slices has read it.  BF16: the
      // activations' arrival; freed by the MMA thread's commit.
      mbar_init(smem_u32(&bar_full[i]), C::kFp4 ? 1 : C::kFullCount);
      mbar_init(smem_u32(&bar_empty[i]), C::kFp4 ? 4 * kSPS : 1);
    }
    for (int i = 0; i < nx; ++i) {
      mbar_init(smem_u32(&bar_xfull[i]), C::kFullCount);  // TMA: one arrival; gathers: 32 lanes + lane 0
      mbar_init(smem_u32(&bar_xempty[i]), 1);
      mbar_init(smem_u32(&bar_xready[i]), 1);
    }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(smem_u32(&bar_afull[i]), 4);  // one arrival per warp of the slice's warpgroup
      mbar_init(smem_u32(&bar_aempty[i]), 1);
    }
    mbar_init(smem_u32(&bar_accum), 1);
    mbar_init(smem_u32(&bar_inbox), 1);
    mbar_init(smem_u32(&bar_red_ready), S);
    mbar_init(smem_u32(&bar_red_done), S);
    if (C::kPush && S > 1) {
      // every rank sends its partials of my rows for all tokens
      const int unit = feature_unit<kMode>(wk);
      const int R = (unit + static_cast<int>(S) - 1) / static_cast<int>(S);
      const int mine = max(0, min(R, unit - static_cast<int>(rank) * R)) * (128 / unit);
      mbar_arrive_expect_tx(smem_u32(&bar_inbox), S * kNT * mine * 4);
    }
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&s_tmem), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (S > 1) {
    if (C::kPush) cluster_arrive_relaxed();  // paired with a wait before the first remote access
    else cluster_sync();
  }
  // Let the next kernel in the stream start its own prologue (weight
  // prefetch) while this grid runs.  (gate_up routed CTAs have already waited
  // for the router, so a dependent kernel that reads ids early is safe.)
  if (tid == 0) pdl_launch_dependents();

  const CtaWork& wk = s_work;
  const bool active = wk.active != 0;
  const uint32_t tmem = s_tmem;
  const int nst = stage_count(wk);
  const int nslices = active ? (wk.k_end - wk.k_begin + kSliceK - 1) / kSliceK : 0;  // 128-K slices (NVFP4)
  // Output rows are reduced per feature unit: a paired tile's feature o lives
  // in rows o and o + 64, so those rows go to the same cluster rank.
  const int unit = feature_unit<kMode>(wk);
  const int R = (unit + static_cast<int>(S) - 1) / static_cast<int>(S);  // features reduced per rank
  const int f_lo = static_cast<int>(rank) * R;
  const int f_hi = min(unit, f_lo + R);
  const int mine = max(0, f_hi - f_lo) * (128 / unit);  // rows this rank owns

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------------ producer
    // The first stages, issued after the CTA barrier so the other warps need
    // not wait for the copies' issue (~2.4 us for three stages of 128-row
    // tiles, measured at a CTA's start; the block barrier held every warp
    // for it when they were issued before).  Still before the wait for the
    // previous grid (gate_up routed CTAs: resolve_work already waited).
    if (lane == 0) {
      pre = min(nst, nstages);
      for (int s = 0; s < pre; ++s) issue_weights(wk, s);
    }
    pdl_wait();
    pre = __shfl_sync(0xFFFFFFFFu, pre, 0);
    if constexpr (C::kFp4) {
      // Weight stages as their slots free up: a stage's slot once the
      // dequant warps have read the stage that held it.
      if (lane == 0) {
        for (int s = pre; s < nst && !s_abort; ++s) {
          if (s >= nstages &&
              !mbar_wait_sleepy(smem_u32(&bar_empty[s % nstages]), ((s / nstages) & 1) ^ 1, p.err, 64)) {
            s_abort = 1;
            break;
          }
          issue_weights(wk, s);
        }
      }
    } else {
      // BF16 (dense): weights and activations of a stage share its slot;
      // rows 0..M-1 of x, one TMA box {64 elements, kNT rows} per stage.
      if (lane == 0) {
        for (int s = 0; s < nst && !s_abort; ++s) {
          const int slot = s % nstages;
          const uint32_t st = ring + slot * C::kStageBytes;
          const uint32_t fb = smem_u32(&bar_full[slot]);
          if (s >= pre) {
            if (!mbar_wait_sleepy(smem_u32(&bar_empty[slot]), ((s / nstages) & 1) ^ 1, p.err, 64)) { s_abort = 1; break; }
            issue_weights(wk, s);
          }
          const int k0 = wk.k_begin + s * C::kStageK;
          mbar_arrive_expect_tx(fb, C::kXBytes);
          tma_load_2d(st + C::kXOff, &p.tm_x, k0, 0, fb, pol_x);
        }
      }
    }
  } else if (warp == C::kXWarp) {
    // ------------------------------------------------------------------ activation producer
    // NVFP4: one 128-K slice per slot, issued once the MMAs of the slice
    // that held the slot are done (dense: TMA by lane 0; MoE: cp.async
    // gathers by all lanes).  Activations are read only after the wait for
    // the previous grid.
    if constexpr (C::kFp4) {
      pdl_wait();
      const uint16_t* xb = wk.shared ? p.x2 : p.x;
      for (int q = 0; q < nslices; ++q) {
        const int xs = q % nx;
        if (!__all_sync(0xFFFFFFFFu, !s_abort && (q < nx || mbar_wait_sleepy(smem_u32(&bar_xempty[xs]),
                                                                               ((q / nx) & 1) ^ 1, p.err, 64)))) {
          s_abort = 1;
          break;
        }
        const uint32_t dst0 = xring + xs * C::kXSliceBytes;
        const uint32_t fb = smem_u32(&bar_xfull[xs]);
        const int k0 = wk.k_begin + q * kSliceK;
        if constexpr (C::kXTma) {
          // rows 0..M-1 of x, one TMA box {64 elements, kNT rows, 2 atoms}
          // (rows beyond M and K beyond the slab's end read as zeros)
          if (lane == 0) {
            mbar_arrive_expect_tx(fb, C::kXSliceBytes);
            tma_load_3d(dst0, &p.tm_x, 0, 0, k0 / kSubK, fb, pol_x);
          }
        } else {
          // gathered rows: lane = 16-byte chunk (of 16 per row slice) +
          // 16 x row parity; 128-byte swizzle within each 64-K atom
          const int cc = lane % 16, rh = lane / 16;
          const bool kok = cc * 8 < min(kSliceK, wk.k_end - k0);
          const uint16_t* src_k = xb + k0 + cc * 8;
          const uint32_t dsta = dst0 + (cc / 8) * (kNT * 128);
#pragma unroll 4
          for (int n = rh; n < kNT; n += 2) {
            const bool valid = kok && n < wk.ntok;
            const uint32_t dst = dsta + (n / 8) * 1024 + (n % 8) * 128 + (((cc % 8) ^ (n % 8)) * 16);
            cp_async16(dst, valid ? src_k + wk.xoff[n] : xb, valid ? 16u : 0u);
          }
          cp_async_arrive_noinc(fb);
          if (lane == 0) mbar_arrive(fb);
        }
      }
    }
  } else if (warp == C::kPermWarp) {
    // ------------------------------------------------------------------ activation permute
    // NVFP4, tiles of up to 32 tokens: each landed slice in place into the
    // weight pairs' K order (dequant.cuh), then a proxy fence (the MMAs read
    // it through the async proxy) and one arrival; the MMA warp waits for
    // it.  The single in-order consumer of the slots' landing barriers
    // (parity waits).
    if constexpr (C::kPermSep) {
      const int klen = wk.k_end - wk.k_begin;
      for (int q = 0; q < nslices; ++q) {
        const int xs = q % nx;
        if (!__all_sync(0xFFFFFFFFu,
                        !s_abort && mbar_wait_sleepy(smem_u32(&bar_xfull[xs]), (q / nx) & 1, p.err, 20))) {
          s_abort = 1;
          break;
        }
        const int natoms = min(kSliceK, klen - q * kSliceK) / kSubK;  // 1 or 2
        for (int v = 0; v < natoms; ++v) {
          const uint32_t xa = xring + xs * C::kXSliceBytes + v * (kNT * 128);
#pragma unroll 4
          for (int c = lane; c < kNT * 8; c += 32) sts128(xa + c * 16, perm_x8(lds128(xa + c * 16)));
        }
        fence_proxy_async_smem();  // the permuted activations, before the MMAs read them
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_xready[xs]));
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    // One warp consumes the slots in slice order (the slot barriers' parity
    // waits rely on a single in-order consumer); the dequant warpgroups never
    // wait on an issue.  The whole warp runs the loop and waits; one elected
    // lane issues a slot's MMAs, unrolled, with the shared-memory descriptors
    // stepped by constants (issued from a loop that lane 0 runs alone,
    // building each descriptor, an MMA costs its thread ~300 cycles instead
    // of ~25).  NVFP4: per 128-K slice (a ring slot of tensor memory, filled
    // by one warpgroup) 8 MMAs of K = 16, one commit that frees the tensor
    // memory slot and one that frees the slice's activation slot.  BF16: both
    // operands in shared memory, 4 MMAs per 64-K stage and a commit that
    // frees the stage.
    if (active) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kNT);
      const int klen = wk.k_end - wk.k_begin;
      const uint32_t acc = tmem;
      if constexpr (C::kFp4) {
        for (int q = 0; q < nslices; ++q) {
          const int a = q % kNS;
          if (!__all_sync(0xFFFFFFFFu, !s_abort && mbar_wait(smem_u32(&bar_afull[a]), (q / kNS) & 1, p.err) &&
                                           (!C::kPermSep ||
                                            mbar_wait(smem_u32(&bar_xready[q % nx]), (q / nx) & 1, p.err)))) {
            s_abort = 1;
            break;
          }
          tc_fence_after();
          // the slice's two 64-K activation atoms
          const uint32_t xs = xring + (q % nx) * C::kXSliceBytes;
          const uint64_t b0 = sdesc_sw128(xs), b1 = sdesc_sw128(xs + kNT * 128);
          const bool full = klen - q * kSliceK >= kSliceK;  // else the last slice, 64 K
          const uint32_t a_tmem = tmem + C::kAccCols + a * C::kSlotCols;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              if (kk < 4 || full)  // +32 bytes of K = +2 in the descriptor's address field
                mma_ts(acc, a_tmem + kk * 8, (kk < 4 ? b0 : b1) + 2 * (kk % 4), idesc, (q > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(smem_u32(&bar_aempty[a]));
            mma_commit(smem_u32(&bar_xempty[q % nx]));
          }
          __syncwarp();
        }
      } else {
        for (int s = 0; s < nst; ++s) {
          const int slot = s % nstages;
          const uint32_t st = ring + slot * C::kStageBytes;
          if (!__all_sync(0xFFFFFFFFu, !s_abort && mbar_wait(smem_u32(&bar_full[slot]), (s / nstages) & 1, p.err))) {
            s_abort = 1;
            break;
          }
          tc_fence_after();
          const uint64_t da = sdesc_sw128(st), db = sdesc_sw128(st + C::kXOff);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ss(acc, da + 2 * kk, db + 2 * kk, idesc, (s > 0 || kk > 0) ? 1u : 0u);
            mma_commit(smem_u32(&bar_empty[slot]));
          }
          __syncwarp();
        }
      }
      if (elect_one()) mma_commit(smem_u32(&bar_accum));
      __syncwarp();
    }
  } else if (active) {
    // ------------------------------------------------------------------ dequant warpgroups
    if constexpr (C::kFp4) {
      const int w = warp / 4;   // warpgroup: slices q = w, w + kW, ...
      const int i = tid % 128;  // row in the tile
      const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
      const int b = wk.paired ? i / 64 : 0;  // box of row i
      const int r = wk.srow[b] + (wk.paired ? i % 64 : i);
      const int gslot = b == 0 ? 0 : 1 + (r / 128 - wk.srow[1] / 128);  // smem scale group of row i
      const uint32_t sf_row_off = C::kWTileBytes + gslot * 2048 + (r % 32) * 16 + ((r % 128) / 32) * 4;
      const uint32_t w_row_off = (i / 8) * 1024 + (i % 8) * 128;
      const uint32_t i8 = i % 8;
      const int klen = wk.k_end - wk.k_begin;
      int cur = -1;  // ring stage whose full barrier this warp has passed
      for (int q = w; q < nslices; q += kW) {
        const int s = q / kSPS, u2 = q % kSPS;
        const int slot = s % nstages;
        const uint32_t st = ring + slot * wstage;
        const uint32_t xs = xring + (q % nx) * C::kXSliceBytes;
        const int a = q % kNS;
        // Waits are bounded and made uniform over the warp (tcgen05.st is
        // warp-collective); a warp that gives up leaves the loop, and the
        // MMA thread's wait on its slot then times out as well.  Each wait
        // comes as late as the work allows: codes and scales are loaded and
        // the stage released first, the first 32 weights dequantized before
        // the tensor-memory slot is waited for.  Tiles of up to 32 tokens:
        // the activations are the permute warp's, these warps never wait
        // for them.  Larger tiles: the warps permute the slice's activations
        // after the tensor-memory slot's wait -- a parity wait on the
        // activation slot is sound only once its previous fill (slice q - nx)
        // is known to have landed, which this warpgroup saw itself when nx
        // is even (the slot holds only its slices) and which the tensor-
        // memory slot's wait implies when nx = kSlots = 3 (slice q - 3
        // consumed).
        bool ok = !s_abort;
        if (ok && s != cur) {
          ok = mbar_wait_sleepy(smem_u32(&bar_full[slot]), (s / nstages) & 1, p.err, 20);
          cur = s;
        }
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          s_abort = 1;
          break;
        }
        const int natoms = min(kSliceK, klen - q * kSliceK) / kSubK;  // 1 or 2
        uint4 qc[2][2];
        uint32_t sw[2] = {0u, 0u};
        uint32_t dep = 0;
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          if (v < natoms) {
            const int u = 2 * u2 + v;  // 64-K atom of the stage
            qc[v][0] = lds128(st + w_row_off + (((2 * u) ^ i8) * 16));
            qc[v][1] = lds128(st + w_row_off + (((2 * u + 1) ^ i8) * 16));
            sw[v] = lds32(st + sf_row_off + u * 512);
            dep ^= qc[v][0].x ^ qc[v][0].y ^ qc[v][0].z ^ qc[v][0].w ^ qc[v][1].x ^ qc[v][1].y ^ qc[v][1].z ^
                   qc[v][1].w ^ sw[v];
          }
        }
        // every lane's loads have returned (dep consumes them) before lane 0
        // releases this warp's share of the stage
        asm volatile("" ::"r"(dep) : "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_empty[slot]));
        uint32_t sc[2][4];
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          scale_pair_to_bf16x2(sw[v] & 0xFFFFu, sc[v][0], sc[v][1]);
          scale_pair_to_bf16x2(sw[v] >> 16, sc[v][2], sc[v][3]);
        }
        uint32_t o[16];
        dequant32_perm(qc[0][0], sc[0][0], sc[0][1], o);
        if (!__all_sync(0xFFFFFFFFu,
                        !s_abort && mbar_wait_sleepy(smem_u32(&bar_aempty[a]), ((q / kNS) & 1) ^ 1, p.err, 20))) {
          s_abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t col0 = tmem + lane_base + C::kAccCols + a * C::kSlotCols;
        tmem_st16(col0, o);
        dequant32_perm(qc[0][1], sc[0][2], sc[0][3], o);
        tmem_st16(col0 + 16, o);
        if (natoms > 1) {
          dequant32_perm(qc[1][0], sc[1][0], sc[1][1], o);
          tmem_st16(col0 + 32, o);
          dequant32_perm(qc[1][1], sc[1][2], sc[1][3], o);
          tmem_st16(col0 + 48, o);
        }
        if constexpr (!C::kPermSep) {
          if (!__all_sync(0xFFFFFFFFu,
                          !s_abort && mbar_wait_sleepy(smem_u32(&bar_xfull[q % nx]), (q / nx) & 1, p.err, 20))) {
            s_abort = 1;
            break;
          }
          // this warp's share of the slice's activations into the pairs' K order
          for (int v = 0; v < natoms; ++v) {
            const uint32_t xa = xs + v * (kNT * 128);
            for (int c = i; c < kNT * 8; c += 128) sts128(xa + c * 16, perm_x8(lds128(xa + c * 16)));
          }
          fence_proxy_async_smem();  // the permuted activations, before the MMAs read them
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_afull[a]));
      }
    }
  }

  // ==================================================================== epilogue
  __syncwarp();
  if (warp < C::kProducerWarp) {
    const int w = warp / 4;
    const int i = tid % 128;
    const bool ok_acc = active && mbar_wait(smem_u32(&bar_accum), 0, p.err);
    if (!ok_acc && active) s_abort = 1;
    tc_fence_after();
    // warp-uniform: the accumulator reads below are warp-collective
    const bool go = __all_sync(0xFFFFFFFFu, ok_acc && !s_abort);
    const float post = C::kFp4 ? static_cast<float>(1 << kShift) : 1.0f;
    constexpr int kCols = kNT / kW;     // token columns this warpgroup reduces
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    // Row i's owner rank and its index among the owner's rows.
    const int fi = i % unit;
    const int owner = fi / R;
    const int owner_feats = min(R, unit - owner * R);
    const int rr = (i / unit) * owner_feats + (fi - owner * R);
    const int rows_owner = owner_feats * (128 / unit);
    // The accumulator's columns [c, c + 8) of row i.
    auto load_sum = [&](int c, float (&v8)[8]) {
      uint32_t v[8];
      tmem_ld8(tmem + lane_base + c, v);
      tmem_wait_ld();
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) v8[jj] = __uint_as_float(v[jj]);
    };
    // Partials of (token n, row i).  Push mode: the owner of row i receives
    // them from every rank into inbox[src][n][rr]; pull mode: each rank leaves
    // its partials in its own ring as red[n][row] and the owner reads them
    // through DSMEM.
    if constexpr (C::kPush) {
      if (S > 1) cluster_wait();  // all peers' inbox barriers are initialised
      if (go) {
        const uint32_t base = inbox + ((rank * kNT) * rows_owner + rr) * 4;
        const uint32_t rbase = S > 1 ? mapa(base, owner) : base;
        const uint32_t rbar = S > 1 ? mapa(smem_u32(&bar_inbox), owner) : 0u;
#pragma unroll
        for (int c = w * kCols; c < (w + 1) * kCols; c += 8) {
          float v8[8];
          load_sum(c, v8);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const uint32_t off = (c + jj) * rows_owner * 4;
            if (S > 1) st_async_f32(rbase + off, v8[jj] * post, rbar);
            else stsf(rbase + off, v8[jj] * post);
          }
        }
      } else if (active && S > 1) {
        // keep the owners' transaction counts consistent on the abort path
        const uint32_t base = inbox + ((rank * kNT) * rows_owner + rr) * 4;
        const uint32_t rbase = mapa(base, owner);
        const uint32_t rbar = mapa(smem_u32(&bar_inbox), owner);
        for (int c = w * kCols; c < (w + 1) * kCols; ++c) st_async_f32(rbase + c * rows_owner * 4, 0.0f, rbar);
      }
      tc_fence_before();
      if (S > 1) {
        if (!mbar_wait<true>(smem_u32(&bar_inbox), 0, p.err)) s_abort = 1;
      } else {
        epi_sync<kEpiThreads>();
      }
    } else {
      epi_sync<kEpiThreads>();  // every ring stage is consumed: reuse it for partials
      if (go) {
#pragma unroll
        for (int c = w * kCols; c < (w + 1) * kCols; c += 8) {
          float v8[8];
          load_sum(c, v8);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) stsf(ring + ((c + jj) * 128 + i) * 4, v8[jj] * post);
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
    // Sum over the cluster ranks, in rank order, of the partial of (token n,
    // tile row) for a row this rank owns; `lr` is the row's index among mine.
    auto partial = [&](int n, int row, int lr) -> float {
      if constexpr (C::kPush) {
        float acc = 0.0f;
        for (uint32_t src = 0; src < S; ++src) acc += ldsf(inbox + ((src * kNT + n) * mine + lr) * 4);
        return acc;
      } else {
        const uint32_t off = ring + (n * 128 + row) * 4;
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
    const int nf = f_hi - f_lo;  // features this rank owns (per unit)
    if (active && !s_abort && nf > 0) {
      pdl_wait();
      if (unit == 128) {
        // plain tiles: feature = tile row
        const float sc = (kMode == kDenseFp4 || kMode == kDenseBf16)
                             ? (p.gs ? __ldg(p.gs) : 1.0f)
                             : (wk.shared ? __ldg(p.gs) : __ldg(p.alpha + wk.expert));
        uint16_t* dst = (kMode == kMoeDown && wk.shared) ? p.out2 : p.out;
        const int64_t ld = (kMode == kMoeDown && wk.shared) ? p.ldo2 : p.ldo;
        const int nfeat = (kMode == kMoeDown && wk.shared) ? p.shared_n_out : p.n_out;
        for (int it = tid; it < nf * wk.ntok; it += kEpiThreads) {
          const int n = it / nf, lr = it % nf, row = f_lo + lr;
          const int o = wk.out_base + row;
          if (o >= nfeat) continue;
          const int64_t orow = (kMode == kMoeDown) ? wk.orow[n] : n;
          dst[orow * ld + o] = f32_to_bf16_rn(partial(n, row, lr) * sc);
        }
      } else if (kMode == kMoeGateUp && !wk.shared) {
        // routed [up; gate] group: feature o = up row o, gate row o + 64
        const float al = __ldg(p.alpha + wk.expert);
        for (int it = tid; it < nf * wk.ntok; it += kEpiThreads) {
          const int n = it / nf, lr = it % nf, o = f_lo + lr;
          const int feat = wk.out_base + o;
          if (feat >= p.n_out) continue;
          const float uu = partial(n, o, lr) * al;
          const float gt = partial(n, o + 64, lr + nf) * al;
          p.out[static_cast<int64_t>(wk.orow[n]) * p.ldo + feat] = f32_to_bf16_rn(silu_fast(gt) * uu);
        }
      } else {
        // paired tiles: feature o = gate row o, up row o + 64
        const float gs = p.gs ? __ldg(p.gs) : 1.0f;
        uint16_t* dst = (kMode == kMoeGateUp) ? p.out2 : p.out;
        const int64_t ld = (kMode == kMoeGateUp) ? p.ldo2 : p.ldo;
        const int nfeat = (kMode == kMoeGateUp) ? p.shared_n_out : p.n_out;
        for (int it = tid; it < nf * wk.ntok; it += kEpiThreads) {
          const int n = it / nf, lr = it % nf, o = f_lo + lr;
          const int feat = wk.out_base + o;
          if (feat >= nfeat) continue;
          const float G = bf16_to_f32(f32_to_bf16_rn(partial(n, o, lr) * gs));
          const float U = bf16_to_f32(f32_to_bf16_rn(partial(n, o + 64, lr + nf) * gs));
          const int64_t orow = (kMode == kMoeGateUp) ? wk.orow[n] : n;
          dst[orow * ld + feat] = f32_to_bf16_rn(silu_exact(G) * U);
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
        // resets the counter.  The previous grid in the stream may be a
        // down_combine on the same workspace (PDL lets this grid start
        // early): its counting must be over before this call's first
        // arrival, which retags the counter.
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
        moe_combine_tile(p, blockIdx.x * 128, tid, kEpiThreads);
      }
    }
  } else if (C::kPush && S > 1) {
    cluster_wait();  // the producer warp closes its cluster-barrier phase
  }

  // ==================================================================== teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fp4
