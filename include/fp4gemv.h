/*
 * fp4gemv.h -- C ABI of libfp4gemv: NVFP4 (W4A16) small-M GEMV kernels for
 * GB300 (sm_103a).
 *
 * Operations (sources are the pages' titles and sections):
 *   vllm.models.flint.ops.nvfp4_gemv  -- nvfp4_gemv, bf16_gemv, dequantize_rows
 *   vllm.models.flint.ops.linear      -- _dequant_gemm (dequantize + GEMM path),
 *                                        _swizzled_scale_buffer (scale size)
 *   vllm.models.flint.ops.moe_gemv    -- gate_up, down_combine
 *
 * Common conventions
 *   - Every pointer argument is DEVICE memory owned by the caller, unless a
 *     parameter says otherwise.  Nothing is allocated or freed inside the
 *     library.  All launches are asynchronous on `stream`.
 *   - bf16 tensors are row-major with unit inner stride; `ld*` arguments are
 *     row strides in ELEMENTS.
 *   - NVFP4 weight: uint8 [rows, K/2], two E2M1 codes per byte, low nibble
 *     first (element 2j in bits 0..3 of byte j).
 *   - Block scales: float8_e4m3fn bytes, one per 16 consecutive K elements,
 *     in the flat 128x4-swizzled buffer of fp4gemv_scale_bytes(rows, K)
 *     bytes: rows padded to 128, K blocks padded to 4; the scale of (row r,
 *     block kb) sits at byte ((r/128)*(Kbp/4) + kb/4)*512 + (r%32)*16 +
 *     ((r%128)/32)*4 + kb%4, Kbp = roundup(K/16, 4).
 *   - Global scales / alphas are fp32 DEVICE values (no host sync).
 *   - Numerics: weights are dequantized exactly (e2m1 * e4m3 is exact in
 *     bf16); products with bf16 activations are exact; sums are fp32; the
 *     fp32 global scale multiplies the fp32 accumulator; one bf16 rounding.
 *   - `pdl` != 0 launches with programmatic dependent launch: weight and
 *     scale loads start before the previous kernel in the stream finishes;
 *     activations are read and outputs written only after it completes.
 *     Pass 0 after kernels that need the whole GPU to make progress.
 *   - Argument errors are detected on the host before any launch and
 *     returned as a status; nothing is launched then.  Conditions only the
 *     device can see (an expert id out of range, a bounded wait that ran
 *     out) are recorded in a per-device error word read by
 *     fp4gemv_get_device_error(); the affected outputs are left unwritten.
 *   - Alignment: bf16 tensors and row strides 16-byte aligned, uint8 weights
 *     16-byte aligned, scale buffers 4-byte aligned (16-byte for the dense
 *     GEMV), fp32 scalars 4-byte aligned.
 *   - Lifetime: the first call on a device looks up the addresses of the
 *     library's own device-side state (the error word and wait limit, the
 *     scratch of fp4gemv_moe_down_combine_noalloc) and keeps them per device
 *     ordinal for the life of the process; encoded tensor maps are cached
 *     per host thread and buffer.  Do not call the library after
 *     cudaDeviceReset() on a device it has used: the new context would make
 *     those addresses stale.
 */
#ifndef FP4GEMV_H
#define FP4GEMV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP4GEMV_OK = 0,
    FP4GEMV_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad flag  */
    FP4GEMV_ERR_UNSUPPORTED_SHAPE = 2, /* a divisibility / range rule not met    */
    FP4GEMV_ERR_MISALIGNED = 3,        /* a pointer or stride breaks alignment   */
    FP4GEMV_ERR_CUDA = 4,              /* a CUDA runtime / driver call failed    */
    FP4GEMV_ERR_TIMEOUT = 5,           /* device: a bounded wait ran out         */
    FP4GEMV_ERR_BAD_INDEX = 6          /* device: expert id outside [0, E)       */
} fp4gemv_status;

/* Largest token count of the GEMV entry points (the MMA N dimension). */
#define FP4GEMV_MAX_M 128

/* Bytes of a flat 128x4-swizzled scale buffer for a [rows, K] weight:
 * roundup(rows, 128) * roundup(K / 16, 4)  (_swizzled_scale_buffer,
 * vllm.models.flint.ops.linear).  Returns 0 for rows < 1 or K < 16. */
size_t fp4gemv_scale_bytes(int rows, int K);

/* nvfp4_gemv (vllm.models.flint.ops.nvfp4_gemv, nvfp4_gemv):
 *   out[m, n] = bf16(fp32(x[m, :] . dequant(W)[n, :]) * global_scale)
 * x     bf16 [M, ldx] (K used), w uint8 [N, K/2], w_sf flat 128x4 scales,
 * global_scale fp32 [1] (device), out bf16 [M, ldo].
 * silu_mul != 0: W's rows are [gate | up] halves (rows [0, N/2) gate, rows
 *   [N/2, N) up); out[m, i] = bf16(silu(G) * U) for i < N/2 with G, U the
 *   bf16 outputs of the gate and up rows (exact SiLU, one rounding).
 * Shapes: 1 <= M <= FP4GEMV_MAX_M, N % 16 == 0 (N % 32 == 0 with silu_mul),
 *   K % 64 == 0 and K >= 256, ldx >= K, ldo >= N (N/2 with silu_mul). */
fp4gemv_status fp4gemv_nvfp4_gemv(const void* x, int64_t ldx, const uint8_t* w, const uint8_t* w_sf,
                                  const float* global_scale, void* out, int64_t ldo, int M, int N, int K,
                                  int silu_mul, int pdl, cudaStream_t stream);

/* fp4gemv_nvfp4_gemv on a scale buffer padded along K (the zero-copy reuse of
 * another library's scale tensor, vllm.models.flint.ops.linear,
 * _swizzled_scale_buffer): each 128-row group of w_sf holds sf_k_blocks
 * 16-wide K blocks (sf_k_blocks / 4 chunks of 512 bytes) instead of
 * roundup(K / 16, 4); the chunks past roundup(K / 16, 4) are never read.
 * sf_k_blocks: 0 (the exact layout) or a multiple of 4 >= roundup(K/16, 4),
 * else FP4GEMV_ERR_INVALID_ARG.  Everything else as fp4gemv_nvfp4_gemv. */
fp4gemv_status fp4gemv_nvfp4_gemv_padded(const void* x, int64_t ldx, const uint8_t* w, const uint8_t* w_sf,
                                         int sf_k_blocks, const float* global_scale, void* out, int64_t ldo, int M,
                                         int N, int K, int silu_mul, int pdl, cudaStream_t stream);

/* bf16_gemv (vllm.models.flint.ops.nvfp4_gemv, bf16_gemv): same contract
 * with a row-major bf16 weight w [N, K] and global scale 1.
 * Shapes: 1 <= M <= FP4GEMV_MAX_M, N % 16 == 0 (N % 32 with silu_mul),
 *   K % 64 == 0, ldx >= K, ldo >= N (N/2). */
fp4gemv_status fp4gemv_bf16_gemv(const void* x, int64_t ldx, const void* w, void* out, int64_t ldo, int M,
                                 int N, int K, int silu_mul, int pdl, cudaStream_t stream);

/* dequantize_rows (vllm.models.flint.ops.nvfp4_gemv, dequantize_rows):
 *   out[r, k] = bf16(e2m1(code(r, k)) * e4m3(scale(r, k / 16)))  exactly,
 *   global scale not applied.  out bf16 [rows, K].
 * Shapes: rows % 16 == 0, K % 256 == 0 (the pages' assertion). */
fp4gemv_status fp4gemv_dequantize_rows(const uint8_t* w, const uint8_t* w_sf, void* out, int rows, int K,
                                       cudaStream_t stream);

/* fp4gemv_dequantize_rows on a scale buffer padded along K: sf_k_blocks as
 * for fp4gemv_nvfp4_gemv_padded (0 or a multiple of 4 >= K / 16). */
fp4gemv_status fp4gemv_dequantize_rows_padded(const uint8_t* w, const uint8_t* w_sf, int sf_k_blocks, void* out,
                                              int rows, int K, cudaStream_t stream);

/* Dequantize + GEMM path (vllm.models.flint.ops.linear, _dequant_gemm):
 *   w_bf16 = dequantize_rows(w, w_sf);  out = bf16(fp32(x @ w_bf16^T) * gs)
 * with the global scale applied to the fp32 accumulator.  w_bf16 is a
 * caller-owned bf16 [N, K] buffer that receives the dequantized weight.
 * Shapes: as fp4gemv_nvfp4_gemv without silu_mul, plus N % 16 == 0 and
 *   K % 256 == 0 (dequantize_rows). */
fp4gemv_status fp4gemv_dequant_gemm(const void* x, int64_t ldx, const uint8_t* w, const uint8_t* w_sf,
                                    const float* global_scale, void* w_bf16, void* out, int64_t ldo, int M,
                                    int N, int K, int pdl, cudaStream_t stream);

/* ---- W4A4 path (vllm.model_executor.kernels.linear.nvfp4.flashinfer, the
 * W4A4 kernels' apply_weights: x_fp4, x_blockscale = scaled_fp4_quant(x,
 * input_global_scale_inv); out = the NVFP4 x NVFP4 GEMM with alpha).  The
 * pages name the quantiser but not its arithmetic; this library's reading,
 * per row m and 16-value block, in binary32 with round-to-nearest-even:
 *   s = (max |x| / 6) * gsi;  sf = nearest finite E4M3 of s (ties to even,
 *   saturating at 448);  codes = nearest E2M1 of x * (gsi / e4m3(sf)) (ties
 *   to the even code, saturating at 6, zero stored as +0; all 0 if sf = 0).
 * The NVFP4 activation tensor has the weights' format: x_fp4 uint8
 * [M, K / 2] (element 2j in the low nibble of byte j), x_sf the flat 128x4
 * layout of fp4gemv_scale_bytes(M, K) bytes (padding bytes written 0).
 * The GEMM: out[m, n] = bf16(fp32(sum_k xq[m, k] * wq[n, k]) * alpha[0]),
 * xq = e2m1 * e4m3 of the activations, wq of the weights (alpha = the
 * activation's and the weight's global scales multiplied).  It runs on this
 * library's NVFP4 GEMV / GEMM kernels over the exact bf16 dequantisation of
 * the activations (every e2m1 * e4m3 product is exact in bf16), in launches
 * of at most FP4GEMV_MAX_M rows; the block-scaled FP4 tensor-core MMA is not
 * used. */

/* Bytes of the bf16 scratch fp4gemv_w4a4_gemm / fp4gemv_w4a4_linear need for
 * M rows of K activations (M * K * 2, rounded up to 16). */
size_t fp4gemv_w4a4_workspace_bytes(int M, int K);

/* scaled_fp4_quant as read above.  x bf16 [M, ldx >= K] (16-byte aligned,
 * ldx * 2 % 16 == 0); gsi fp32 [1] device (> 0, finite; x finite); x_fp4
 * [M, K / 2] (8-byte aligned) and x_sf (fp4gemv_scale_bytes(M, K) bytes)
 * device, written; x_deq: NULL, or bf16 [M, K] device (16-byte aligned)
 * that receives the exact dequantised values e2m1 * e4m3 (no global scale).
 * Shapes: M >= 1, K % 16 == 0.  One launch. */
fp4gemv_status fp4gemv_quantize_act(const void* x, int64_t ldx, const float* gsi, uint8_t* x_fp4, uint8_t* x_sf,
                                    void* x_deq, int M, int K, cudaStream_t stream);

/* The W4A4 GEMM on quantised activations (x_fp4, x_sf as written by
 * fp4gemv_quantize_act) and NVFP4 weights (w, w_sf as for
 * fp4gemv_nvfp4_gemv): the activations are dequantised into `workspace`
 * (fp4gemv_w4a4_workspace_bytes(M, K) bytes, 16-byte aligned, device), then
 * out bf16 [M, ldo >= N] = bf16(fp32(xq @ wq^T) * alpha[0]).  Shapes: M >= 1
 * (any; launches of FP4GEMV_MAX_M rows), N % 16 == 0, K % 64 == 0,
 * K >= 256.  pdl as for fp4gemv_nvfp4_gemv (the GEMM launches). */
fp4gemv_status fp4gemv_w4a4_gemm(const uint8_t* x_fp4, const uint8_t* x_sf, const uint8_t* w, const uint8_t* w_sf,
                                 const float* alpha, void* out, int64_t ldo, int M, int N, int K, void* workspace,
                                 size_t workspace_bytes, int pdl, cudaStream_t stream);

/* Quantisation and GEMM in one call: fp4gemv_quantize_act into x_fp4 / x_sf,
 * whose kernel also writes the exact dequantised activations into
 * `workspace`, then the GEMM of fp4gemv_w4a4_gemm on them (no second pass
 * over the codes).  Arguments and shapes as those two calls; with pdl = 1
 * the quantisation launch is also early (it waits for the previous grid
 * before reading x). */
fp4gemv_status fp4gemv_w4a4_linear(const void* x, int64_t ldx, const float* gsi, const uint8_t* w,
                                   const uint8_t* w_sf, const float* alpha, void* out, int64_t ldo, int M, int N,
                                   int K, uint8_t* x_fp4, uint8_t* x_sf, void* workspace, size_t workspace_bytes,
                                   int pdl, cudaStream_t stream);

/* gate_up (vllm.models.flint.ops.moe_gemv, gate_up), one launch:
 * routed pairs p = t * topk + j (t < M, j < topk), e = ids[p]:
 *   g, u = fp32(x[t] . W1[e] gate / up row) * alpha[e]   (fp32, not rounded)
 *   act[p, i] = bf16(silu(g_i) * u_i)                 (fast sigmoid)
 * shared expert, every token t:
 *   G, U = bf16(fp32(x[t] . Wsh gate / up row) * gssh[0])
 *   sact[t, i] = bf16(silu(G_i) * U_i)                (exact SiLU)
 * x bf16 [M, H]; ids int32 [M, topk]; w1 uint8 [E, 2I, H/2] with rows
 * "[up; gate] in 64-row groups" (stored rows 128g + [0,64) are up rows
 * 64g + [0,64), stored rows 128g + [64,128) the gate rows); w1_sf = E
 * consecutive flat 128x4 buffers of fp4gemv_scale_bytes(2I, H) bytes;
 * alpha fp32 [E]; act bf16 [M*topk, I]; wsh uint8 [2 SI, H/2] ModelOpt
 * [gate; up]; ssh flat 128x4 scales of [2 SI, H]; gssh fp32 [1];
 * sact bf16 [M, SI].
 * Shapes: 1 <= M, 1 <= topk, M * topk <= 1024, H % 64 == 0 and H >= 256,
 *   I % 64 == 0, SI % 64 == 0, E >= 1.  Pairs whose id is outside [0, E) are left
 *   unwritten and raise FP4GEMV_ERR_BAD_INDEX in the device error word. */
fp4gemv_status fp4gemv_moe_gate_up(const void* x, const int32_t* ids, int M, int topk, const uint8_t* w1,
                                   const uint8_t* w1_sf, const float* alpha, int E, int H, int I, void* act,
                                   const uint8_t* wsh, const uint8_t* ssh, const float* gssh, int SI, void* sact,
                                   int pdl, cudaStream_t stream);

/* Scratch bytes fp4gemv_moe_down_combine needs for M tokens, top-k and
 * hidden size H: per-row-tile counters (arrival counts, or the tags of row
 * tiles whose computation gave up) and one work counter of the persistent
 * grid, then the bf16 y_j and y_shared values.  The contents need no initialisation and carry nothing
 * between calls; one workspace serves calls of any shape that fit in it.
 * Calls that may run concurrently on the GPU must not share a workspace. */
size_t fp4gemv_moe_down_combine_workspace_bytes(int M, int topk, int H);

/* down_combine (vllm.models.flint.ops.moe_gemv, down_combine).  When the
 * slab kernel serves the call (fp4gemv_plan_moe_down_slab; one CTA per item
 * or, beyond one wave, the persistent grid) it is followed by a small
 * combine kernel on the same stream (two launches);
 * otherwise one launch combines in its last CTAs:
 *   y_j  = bf16(fp32(act[t*topk+j] . W2[e_j] row h) * alpha2[e_j])
 *   y_sh = bf16(fp32(sact[t] . Wsd row h) * gssd[0])
 *   out[t, h] = bf16(bf16(sum_j tw[t, j] * y_j) + y_sh)   (fp32 sum, j order)
 * act bf16 [M*topk, I]; ids int32 [M, topk]; tw fp32 [M, topk];
 * w2 uint8 [E, H, I/2]; w2_sf = E flat buffers of fp4gemv_scale_bytes(H, I);
 * alpha2 fp32 [E]; sact bf16 [M, SI]; wsd uint8 [H, SI/2]; ssd flat scales
 * of [H, SI]; gssd fp32 [1]; out bf16 [M, H].
 * workspace: fp4gemv_moe_down_combine_workspace_bytes(M, topk, H) bytes,
 * 16-byte aligned, no initialisation needed (see above).
 * Shapes: 1 <= M, 1 <= topk, M * topk <= 1024, H % 64 == 0,
 *   I % 64 == 0 and I >= 256, SI % 64 == 0 and SI >= 256.  Tokens with an id outside [0, E) are left
 *   unwritten and raise FP4GEMV_ERR_BAD_INDEX. */
fp4gemv_status fp4gemv_moe_down_combine(const void* act, const int32_t* ids, const float* tw, int M, int topk,
                                        const uint8_t* w2, const uint8_t* w2_sf, const float* alpha2, int E, int H,
                                        int I, const void* sact, const uint8_t* wsd, const uint8_t* ssd,
                                        const float* gssd, int SI, void* out, void* workspace,
                                        size_t workspace_bytes, int pdl, cudaStream_t stream);

/* Size of the scratch array behind fp4gemv_moe_down_combine_noalloc: 8 MiB
 * of device memory per GPU that loads the library, held until exit. */
#define FP4GEMV_NOALLOC_SCRATCH_BYTES (8u << 20)

/* down_combine for callers that cannot allocate device memory: the pages
 * have no counterpart of this entry point.  Same arguments, layouts and
 * result as fp4gemv_moe_down_combine, minus the workspace: the scratch is a
 * fixed FP4GEMV_NOALLOC_SCRATCH_BYTES device array inside the library, so
 * nothing is allocated or freed by the call.  For callers whose device
 * memory is planned once at start-up (a serving process that must not
 * allocate on the request path, where cudaMalloc can also synchronize the
 * device) or that own no allocator (a plug-in that only receives tensors).
 * Returns FP4GEMV_ERR_UNSUPPORTED_SHAPE when
 * fp4gemv_moe_down_combine_workspace_bytes(M, topk, H) exceeds
 * FP4GEMV_NOALLOC_SCRATCH_BYTES.  The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture.  All calls
 * share the one array: calls that overlap on the GPU race on it. */
fp4gemv_status fp4gemv_moe_down_combine_noalloc(const void* act, const int32_t* ids, const float* tw, int M,
                                                int topk, const uint8_t* w2, const uint8_t* w2_sf,
                                                const float* alpha2, int E, int H, int I, const void* sact,
                                                const uint8_t* wsd, const uint8_t* ssd, const float* gssd, int SI,
                                                void* out, int pdl, cudaStream_t stream);

/* Synchronizes `stream`, then returns and clears the device error word of
 * the current device: FP4GEMV_OK, FP4GEMV_ERR_TIMEOUT or
 * FP4GEMV_ERR_BAD_INDEX (timeout reported first when both are set).
 * Returns FP4GEMV_ERR_CUDA if the synchronization itself fails. */
fp4gemv_status fp4gemv_get_device_error(cudaStream_t stream);

/* Wait limit of the kernels' bounded waits on the current device, in ns
 * (0 restores the built-in 2 s).  A wait that runs out records
 * FP4GEMV_ERR_TIMEOUT in the device error word and the kernel winds down,
 * leaving its outputs unwritten.  Synchronous; affects launches made after
 * it returns.  FP4GEMV_ERR_CUDA if the device copy fails. */
fp4gemv_status fp4gemv_set_wait_limit_ns(uint64_t ns);

/* Test hook for the timeout path (no counterpart on the pages): from now on
 * the producers of the dense NVFP4 GEMV for 1 .. 16 tokens, and of
 * fp4gemv_moe_down_combine on the slab kernel (1 .. 64 tokens, where its plan applies),
 * issue nothing at all -- no copy, no arrival -- for the 256-K ring stage
 * with this index of every CTA (down_combine: counted over the CTA's row
 * tiles, and on the persistent grid over its items, in turn, the item
 * stream's end counting as one stage), so the consumers' bounded wait for it runs out with no
 * copy in flight; -1 (the default) turns it off.  A process-wide host
 * setting read at each of those launches; for tests only.
 * FP4GEMV_ERR_INVALID_ARG for stage < -1. */
fp4gemv_status fp4gemv_debug_skip_stage(int stage);

/* Static, human-readable name of a status code. */
const char* fp4gemv_status_string(fp4gemv_status status);

/* Number of kernel launches the library has issued in this process (all
 * devices).  Lets a caller count the launches inside a timed region. */
uint64_t fp4gemv_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FP4GEMV_H */
