/*
 * fp4gemv_plan.h -- the launch plans libfp4gemv's dense GEMVs use, as
 * host-only functions: the slab kernel's (NVFP4, large weights at M <= 4),
 * the register-fed kernel's (NVFP4, M <= 16 otherwise) and the tcgen05
 * kernel's (NVFP4 M > 16, BF16 weights).
 *
 * Operation: the grid decomposition of nvfp4_gemv (vllm.models.flint.ops.
 * nvfp4_gemv, nvfp4_gemv): which tile height and K split the library
 * launches for a weight of N x K (with or without silu_mul) on a GPU whose
 * co-resident CTA counts are given.  fp4gemv_nvfp4_gemv computes exactly
 * this plan (with the counts it queries from the device) before launching,
 * so the planning can be checked without a GPU.
 */
#ifndef FP4GEMV_PLAN_H
#define FP4GEMV_PLAN_H

#include "fp4gemv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int tile_rows;     /* weight rows per CTA tile: 96, 112 or 128 (silu_mul: half gate, half up rows) */
  int split;         /* CTAs per cluster along K (1, 2, 4 or 8) */
  int ctas;          /* grid size: tiles x split */
  int scale_groups;  /* 128-row scale groups a ring stage reserves room for (1 .. 4) */
} fp4gemv_rf_plan;

/* Plan of fp4gemv_nvfp4_gemv for M <= 16 when fp4gemv_plan_slab has no
 * plan.
 *   N, K, silu_mul: as fp4gemv_nvfp4_gemv (same shape rules).
 *   sms:  streaming multiprocessors of the GPU (152 on GB300).
 *   cap:  HOST array of 9 ints; cap[s] (s = 1 .. 8) is the number of CTAs
 *         that fit on the GPU at once in whole clusters of s CTAs (cap[0] is
 *         ignored).
 *   out:  HOST pointer, filled on success.
 * Returns FP4GEMV_ERR_INVALID_ARG for null pointers or sms < 1,
 * FP4GEMV_ERR_UNSUPPORTED_SHAPE for shapes fp4gemv_nvfp4_gemv rejects. */
fp4gemv_status fp4gemv_plan_rf(int N, int K, int silu_mul, int sms, const int* cap, fp4gemv_rf_plan* out);

typedef struct {
  int row_blocks;     /* 16-row blocks per consumer warp: 1 or 2 */
  int warps;          /* consumer warps per CTA: 2 or 4 (the CTA adds one producer warp) */
  int tile_rows;      /* weight rows per CTA tile: 16 x row_blocks x warps (silu_mul: half gate, half up) */
  int split;          /* CTAs per cluster along K (1 .. 16) */
  int ctas;           /* grid size: tiles x split */
  int k_slab;         /* K elements per cluster rank, a multiple of 64 */
  int stages;         /* weight ring stages of 256 K */
  int slab_bytes;     /* shared memory holding the CTA's activations */
  int ctas_per_sm;    /* CTAs an SM runs at once with this shared memory, threads and registers */
  size_t smem_bytes;  /* dynamic shared memory per CTA */
} fp4gemv_slab_plan;

/* Plan of fp4gemv_nvfp4_gemv on the slab kernel (the kernel that keeps each
 * CTA's activations in shared memory).  No GPU is needed.
 *   M, N, K, silu_mul: as fp4gemv_nvfp4_gemv (same shape rules).
 *   sms:  streaming multiprocessors of the GPU (152 on GB300).
 *   regs: HOST array of 2 ints, registers per thread of the kernel with 1
 *         and with 2 row blocks per warp (they bound the CTAs per SM).
 *   out:  HOST pointer, filled on success.
 * Applies to 1 <= M <= 4 and weights of at least 1.2 x sms tiles of 128
 * rows (e.g. the gate_up projections of Llama-3-8B / 70B): on smaller grids
 * and more tokens the register-fed kernel was as fast or faster.
 * Returns FP4GEMV_ERR_INVALID_ARG for null pointers, sms < 1 or a flag
 * outside {0, 1}; FP4GEMV_ERR_UNSUPPORTED_SHAPE for shapes the GEMV rejects
 * and for calls the slab kernel does not serve (they run on the kernel
 * fp4gemv_plan_rf describes). */
fp4gemv_status fp4gemv_plan_slab(int M, int N, int K, int silu_mul, int sms, const int* regs, fp4gemv_slab_plan* out);

typedef struct {
  int split;          /* split form: CTAs per cluster along H (1, 2, 4 or 8); grouped form: 1 */
  int k_slab;         /* H elements per cluster rank, a multiple of 64 (grouped form: H) */
  int tiles_per_cta;  /* 0: split form, one tile per CTA; else grouped form, the most tiles one CTA takes */
  int groups;         /* grid columns: tiles x split (split form) or tile groups (grouped form) */
  int chunk_pairs;    /* most (token, expert) pairs one routed CTA computes (1, 2 or 4) */
  int columns;        /* grid rows: M * topk routed pair columns + the shared expert's token chunks */
  int tiles;          /* 128-row tiles per column: max(I / 64, ceil(SI / 64)) */
  int slab_bytes;     /* shared memory holding a CTA's activations */
  int stage_bytes;    /* one weight stage (codes of 128 rows x 256 K, two scale groups) */
  int stages;         /* weight ring stages (2 .. 8) */
  int ctas_per_sm;    /* CTAs per SM the shared memory is sized for (2 or 3) */
  size_t smem_bytes;  /* dynamic shared memory per CTA */
} fp4gemv_moe_slab_plan;

/* Plan of fp4gemv_moe_gate_up on the slab kernel (vllm.models.flint.ops.
 * moe_gemv, gate_up: routed chunks of pairs of one expert and the shared
 * expert's token chunks, the CTA's activations in shared memory).  No GPU
 * is needed.
 *   M, topk, E, H, I, SI: as fp4gemv_moe_gate_up (same shape rules).
 *   sms:  streaming multiprocessors of the GPU (152 on GB300).
 *   regs: registers per thread of the kernel.
 *   out:  HOST pointer, filled on success.
 * Split form, when the CTAs of every expert the call can touch (at most
 * min(M * topk, E) routed chunks of 4 pairs plus the shared expert's) fit
 * one wave at three CTAs per SM with a split of H that leaves each rank at
 * least 256 (one token on the E = 128, top-8, H = 4096, I = SI = 1536 block:
 * a split of two).  Otherwise, up to 64 tokens, the grouped form: the whole
 * H per CTA and T of its column's tiles in turn (T = 1 up to 2 tokens, else
 * 2), many waves of CTAs; chunks of 1 pair up to 2 tokens, 2 below 32, 4
 * from 32 (halved while fewer than two stages fit); three CTAs per SM, two
 * from 32 tokens; as many weight stages as fit (2 .. 8).  From 3 to 31
 * tokens, with n(T, c) = (E (1 - (1 - 1/E)^(M topk)), at least
 * ceil(M topk / c)) + ceil(M / c) expected streaming columns times
 * ceil(tiles / T) and f = n(2, 2) / (3 sms): f < 0.7 with n(2, 4) <= 2 sms
 * takes T = 2, chunks of 4, two CTAs per SM; 0.9 < f <= 1.35 takes T = 1.
 * Returns FP4GEMV_ERR_INVALID_ARG for a null out, sms < 1 or regs < 1;
 * FP4GEMV_ERR_UNSUPPORTED_SHAPE for shapes fp4gemv_moe_gate_up rejects and
 * for calls the slab kernel does not serve (they run on the register-fed
 * kernel, chunks of 8 pairs, or beyond 64 tokens on the tcgen05 kernel). */
fp4gemv_status fp4gemv_plan_moe_slab(int M, int topk, int E, int H, int I, int SI, int sms, int regs,
                                     fp4gemv_moe_slab_plan* out);

typedef struct {
  int tiles_per_cta;  /* most 128-row tiles of H one CTA streams in turn: ceil(tiles / groups) */
  int groups;         /* grid columns along H; group g takes tiles [g tiles / groups, (g + 1) tiles / groups) */
  int columns;        /* grid rows: M * topk routed pair columns + the shared expert's token chunks */
  int chunk_pairs;    /* most (token, expert) pairs one routed CTA (or item) computes (8, or 4) */
  int slab_bytes;     /* shared memory holding a CTA's activation rows (the whole K) */
  int stage_bytes;    /* one weight stage (codes of 128 rows x 256 K, one scale group) */
  int stages;         /* weight ring stages (2 .. 8) */
  int ctas_per_sm;    /* CTAs per SM the ring is sized for (2 or 3) */
  int persistent;     /* 1: a persistent grid of ctas_per_sm x sms CTAs takes the groups x columns items in turn */
  size_t smem_bytes;  /* dynamic shared memory per CTA */
} fp4gemv_moe_down_slab_plan;

/* Plan of fp4gemv_moe_down_combine on the slab kernel (vllm.models.flint.ops.
 * moe_gemv, down_combine: chunks of up to 8 pairs of one expert, each CTA
 * streaming T row tiles of its expert over its resident activation rows and
 * writing each tile's y rows; a second, small kernel then combines them).
 * No GPU is needed.
 *   M, topk, E, H, I, SI: as fp4gemv_moe_down_combine (same shape rules).
 *   sms:  streaming multiprocessors of the GPU (152 on GB300).
 *   regs: registers per thread of the kernel.
 *   out:  HOST pointer, filled on success.
 * Applies to 1 <= M <= 64 when up to 8 activation rows of max(I, SI) and
 * two weight stages fit the CTA's share of the SM's shared memory, and the
 * CTA's T tiles of I hold at least two 256-K stages.  Chunks of 8 pairs (but see below).  With C = (E (1 - (1 - 1/E)^(M topk)), at
 * least ceil(M topk / 8)) + ceil(M / 8) expected streaming columns and
 * n(T) = C ceil(ceil(H / 128) / T) CTAs: T = 1 at two CTAs per SM if
 * n(1) <= 2 sms, else T = 2 at two per SM if n(2) <= 2 sms, else T = 1 at
 * three per SM if 0.9 < n(2) / (3 sms) <= 1.35, else T = 2 at three per SM.
 * When that grid holds more than one wave (n(T) > CTAs per SM x sms), the
 * persistent grid (persistent = 1): three CTAs per SM that take items of T
 * tiles of one column in turn from a counter; chunks of 4 pairs if
 * M topk <= E (C and n(T) taken again with them); T = 4 if
 * n(4) >= 1.6 x 3 sms, else 2 if n(2) is, else 1.  As many weight stages as fit (2 .. 8; on
 * the grid of one CTA per item at most T stage streams of I).  tiles_per_cta
 * reports the largest group, ceil(tiles / groups).
 * Returns FP4GEMV_ERR_INVALID_ARG for a null out, sms < 1 or regs < 1;
 * FP4GEMV_ERR_UNSUPPORTED_SHAPE for shapes fp4gemv_moe_down_combine rejects
 * and for calls the slab kernel does not serve. */
fp4gemv_status fp4gemv_plan_moe_down_slab(int M, int topk, int E, int H, int I, int SI, int sms, int regs,
                                          fp4gemv_moe_down_slab_plan* out);

typedef struct {
  int tokens_tile;    /* MMA N of the tcgen05 kernel: 16, 32, 64 or 128 (covers M) */
  int ctas_per_sm;    /* 2, or 1 when the tile's tensor memory needs more than 256 columns */
  int tiles;          /* CTA tiles along N: 128 features, or 64 with silu_mul */
  int split;          /* CTAs per cluster along K (1 .. 8) */
  int k_slab;         /* K elements per cluster rank, a multiple of 64 */
  int weight_stages;  /* weight ring stages of 256 K (2 .. 8) */
  int act_slots;      /* NVFP4: activation slots of one 128-K slice (2 .. 4); BF16: 0 */
  int scale_slots;    /* NVFP4: 2 KB scale groups per weight stage (1 .. 3) */
  int inbox_in_ring;  /* 1: the split-K inbox reuses the drained ring (one rank) */
  size_t smem_bytes;  /* dynamic shared memory per CTA */
} fp4gemv_tc_plan;

/* Plan of the tcgen05 kernel: fp4gemv_nvfp4_gemv for M > 16, and
 * fp4gemv_bf16_gemv (bf16_weights = 1) for any M.  The launch uses exactly
 * this plan; no GPU is needed to compute it.
 *   M, N, K, silu_mul: as the GEMV call (same shape rules).
 *   bf16_weights: 0 = NVFP4 weights, 1 = BF16 weights.
 *   sms:  streaming multiprocessors of the GPU (152 on GB300).
 *   out:  HOST pointer, filled on success.
 * Returns FP4GEMV_ERR_INVALID_ARG for a null out, sms < 1 or flags outside
 * {0, 1}, FP4GEMV_ERR_UNSUPPORTED_SHAPE for shapes the GEMV rejects and
 * for NVFP4 weights with M <= 16 (the register-fed kernel; see
 * fp4gemv_plan_rf). */
fp4gemv_status fp4gemv_plan_tc(int M, int N, int K, int silu_mul, int bf16_weights, int sms, fp4gemv_tc_plan* out);

#ifdef __cplusplus
}
#endif

#endif /* FP4GEMV_PLAN_H */
