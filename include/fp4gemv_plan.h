/*
 * fp4gemv_plan.h -- the launch plan libfp4gemv's dense NVFP4 GEMV uses for
 * M <= 16 (the register-fed kernel), as a host-only function.
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

/* Plan of fp4gemv_nvfp4_gemv for M <= 16.
 *   N, K, silu_mul: as fp4gemv_nvfp4_gemv (same shape rules).
 *   sms:  streaming multiprocessors of the GPU (152 on GB300).
 *   cap:  HOST array of 9 ints; cap[s] (s = 1 .. 8) is the number of CTAs
 *         that fit on the GPU at once in whole clusters of s CTAs (cap[0] is
 *         ignored).
 *   out:  HOST pointer, filled on success.
 * Returns FP4GEMV_ERR_INVALID_ARG for null pointers or sms < 1,
 * FP4GEMV_ERR_UNSUPPORTED_SHAPE for shapes fp4gemv_nvfp4_gemv rejects. */
fp4gemv_status fp4gemv_plan_rf(int N, int K, int silu_mul, int sms, const int* cap, fp4gemv_rf_plan* out);

#ifdef __cplusplus
}
#endif

#endif /* FP4GEMV_PLAN_H */
