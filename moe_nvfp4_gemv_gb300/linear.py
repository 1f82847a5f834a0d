"""Dense linear layers that route each call by its token count.

The dispatch of vllm.models.flint.ops.linear (FlintNvFp4LinearKernel.
apply_weights, FlintBf16LinearMethod.apply, _use_gemv, _dequant_gemm,
gate_up_silu_mul) over this library's kernels:

* NVFP4 weights (``NvFp4Linear``): a call of M tokens (the input flattened
  to [M, K]) runs the small-M GEMV (``fp4gemv.nvfp4_gemv``) while
  ``M < dequant_min_m``; from ``dequant_min_m`` tokens it dequantizes the
  weight to BF16 and runs a GEMM with the global scale as alpha on the fp32
  accumulator -- this library's tensor-core GEMM up to ``MAX_M`` tokens
  (``fp4gemv.dequant_gemm``), cuBLAS beyond or on a scale buffer padded along
  K (``torch.addmm`` with BF16 reduced-precision reductions off, alpha the
  host copy of the global scale, as the page does).
* BF16 weights (``Bf16Linear``): ``fp4gemv.bf16_gemv`` up to
  ``gemv_max_m`` tokens, cuBLAS (``torch.nn.functional.linear``) beyond.
* Fused gate/up projections (``[gate | up]`` halves of N): ``gate_up_silu_mul``
  returns ``bf16(silu(G) * U)`` from one GEMV for small M, else None (the
  caller runs the linear and its own silu_and_mul).
* W4A4 (``NvFp4W4A4Linear``; the flashinfer page's W4A4 kernels,
  apply_weights): the activations are quantised to NVFP4
  (``fp4gemv.quantize_act``) and multiplied with the NVFP4 weight, alpha on
  the fp32 accumulator -- ``fp4gemv.w4a4_linear`` up to ``MAX_M`` tokens;
  beyond, the quantiser's exact dequantised activations times the
  dequantized weight on cuBLAS (``torch.addmm``, alpha the host copy), one
  weight pass instead of one per 128 tokens.

The pages route by tuned tables (``pick_nt`` / ``tuned``, contents not
printed).  Here the library accepts every valid shape and picks its launch
shape itself, so ``gemv_tile`` answers only which token tile a call uses and
``DEQUANT_MIN_M`` is the measured crossover: on GB300, N = K = 8192, the GEMV
was faster than dequantize + GEMM at every M up to 128 (43.5 vs 64.6 us at
M = 128), so the GEMV serves every M it supports and the dequantize + GEMM
path starts past it.
"""
from __future__ import annotations

import torch

from . import fp4gemv

MAX_M = fp4gemv.MAX_M
# First token count routed to dequantize + GEMM (the GEMV is faster up to MAX_M).
DEQUANT_MIN_M = MAX_M + 1
# Largest token count the BF16 GEMV takes by default (cuBLAS beyond).
# Measured on GB300 against torch.matmul (L2-cold, CUDA-graph replay), us at
# M = 1 / 8 / 32 / 128: o_proj 4096x4096 GEMV 7.6 / 7.6 / 9.1 / 20.0 vs cuBLAS
# 8.6 / 8.7 / 9.1 / 8.2; down 4096x14336 18.9 / 19.8 / 20.9 / 31.7 vs
# 21.4 / 21.2 / 22.1 / 25.1; gate_up 28672x4096 35.3 / 37.2 / 42.1 / 58.9 vs
# 36.1 / 35.9 / 36.5 / 41.6; qkv 6144x4096 11.0 / 11.3 / 13.2 / 25.6 vs
# 9.7 / 9.6 / 9.7 / 10.0.  The GEMV wins mostly up to 8 tokens.
BF16_GEMV_MAX_M = 8


def gemv_tile(m: int) -> int | None:
    """Token tile the GEMV uses for ``m`` tokens (the MMA N it covers): 8 or
    16 for the register-fed kernels, 16 .. 128 for the tensor-core kernel;
    None when the GEMV does not take ``m`` (the analogue of ``pick_nt``)."""
    if m < 1 or m > MAX_M:
        return None
    if m <= 8:
        return 8
    if m <= 16:
        return 16
    t = 32
    while t < m:
        t *= 2
    return t


class NvFp4Linear(torch.nn.Module):
    """y = bf16(fp32(x @ dequant(W)^T) * global_scale), routed by token count.

    weight: uint8 [N, K/2] (two E2M1 codes per byte, low nibble first);
    weight_scale: the 128x4-swizzled E4M3 block scales of [N, K] (uint8 or
    float8_e4m3fn), as the flat buffer or as another library's strided view
    of it (used without a copy, vllm.models.flint.ops.linear,
    _swizzled_scale_buffer); ``sf_k_blocks``: 16-wide K blocks per 128-row
    group when the buffer is padded along K (0: roundup(K / 16, 4));
    global_scale: fp32 [1] on the weight's device.  ``pdl``: launch the GEMV
    with programmatic dependent launch (pass False after kernels that need
    the whole GPU).  ``dequant_min_m``: first token count routed to
    dequantize + GEMM."""

    def __init__(self, weight: torch.Tensor, weight_scale: torch.Tensor, global_scale: torch.Tensor,
                 pdl: bool = True, dequant_min_m: int = DEQUANT_MIN_M, sf_k_blocks: int = 0):
        super().__init__()
        if weight.dtype != torch.uint8 or weight.dim() != 2 or not weight.is_contiguous():
            raise ValueError("weight must be a contiguous uint8 [N, K/2] tensor")
        N, K = weight.shape[0], weight.shape[1] * 2
        sf = fp4gemv.flat_scale_buffer(weight_scale)
        kbp = sf_k_blocks or (K // 16 + 3) // 4 * 4
        need = (N + 127) // 128 * 128 * kbp
        if sf.numel() < need:
            raise ValueError(f"weight_scale must hold at least {need} bytes (128x4-swizzled [N, {kbp}] blocks)")
        if global_scale.dtype != torch.float32 or global_scale.numel() != 1:
            raise ValueError("global_scale must be one float32 value")
        self.register_buffer("weight", weight, persistent=False)
        self.register_buffer("weight_scale", sf, persistent=False)
        self.register_buffer("global_scale", global_scale.reshape(1), persistent=False)
        self.global_scale_host = float(global_scale.reshape(()).item())  # alpha of the cuBLAS path
        self.out_features, self.in_features = N, K
        self.pdl = bool(pdl)
        self.dequant_min_m = int(dequant_min_m)
        self.sf_k_blocks = int(sf_k_blocks)

    def route(self, m: int) -> str:
        """'empty', 'gemv' or 'dequant_gemm' for a call of ``m`` tokens."""
        if m == 0:
            return "empty"
        if m >= self.dequant_min_m or gemv_tile(m) is None:
            return "dequant_gemm"
        return "gemv"

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        x2 = x.reshape(-1, x.shape[-1])
        m = x2.shape[0]
        route = self.route(m)
        if route == "empty":
            return x2.new_empty(*x.shape[:-1], self.out_features)
        if route == "gemv":
            out = fp4gemv.nvfp4_gemv(x2, self.weight, self.weight_scale, self.global_scale, pdl=self.pdl,
                                     sf_k_blocks=self.sf_k_blocks)
        else:
            out = self._dequant_gemm(x2)
        return out.view(*x.shape[:-1], self.out_features)

    def _dequant_gemm(self, x2: torch.Tensor) -> torch.Tensor:
        if x2.shape[0] <= MAX_M and not self.sf_k_blocks:
            return fp4gemv.dequant_gemm(x2, self.weight, self.weight_scale, self.global_scale)
        # past MAX_M tokens (or on a padded scale buffer): dequantize, then cuBLAS
        w = fp4gemv.dequantize_rows(self.weight, self.weight_scale, sf_k_blocks=self.sf_k_blocks)
        out = torch.empty(x2.shape[0], self.out_features, dtype=torch.bfloat16, device=x2.device)
        matmul = torch.backends.cuda.matmul
        prev = matmul.allow_bf16_reduced_precision_reduction
        matmul.allow_bf16_reduced_precision_reduction = False  # fp32 split-K sums
        try:
            torch.addmm(out, x2, w.t(), beta=0, alpha=self.global_scale_host, out=out)
        finally:
            matmul.allow_bf16_reduced_precision_reduction = prev
        return out

    def gate_up_silu_mul(self, x: torch.Tensor) -> torch.Tensor | None:
        """bf16(silu(G) * U) of the [gate | up] halves in one GEMV when the
        GEMV takes this call, else None."""
        if x.dim() != 2 or self.out_features % 32 != 0 or self.route(x.shape[0]) != "gemv":
            return None
        return fp4gemv.nvfp4_gemv(x, self.weight, self.weight_scale, self.global_scale, silu_mul=True, pdl=self.pdl,
                                  sf_k_blocks=self.sf_k_blocks)


class Bf16Linear(torch.nn.Module):
    """y = bf16(fp32(x @ W^T)) for a row-major bf16 [N, K] weight: the GEMV up
    to ``gemv_max_m`` tokens, cuBLAS beyond."""

    def __init__(self, weight: torch.Tensor, pdl: bool = True, gemv_max_m: int = BF16_GEMV_MAX_M):
        super().__init__()
        if weight.dtype != torch.bfloat16 or weight.dim() != 2 or not weight.is_contiguous():
            raise ValueError("weight must be a contiguous bf16 [N, K] tensor")
        self.register_buffer("weight", weight, persistent=False)
        self.out_features, self.in_features = weight.shape
        self.pdl = bool(pdl)
        self.gemv_max_m = min(int(gemv_max_m), MAX_M)

    def route(self, m: int) -> str:
        if m == 0:
            return "empty"
        return "gemv" if m <= self.gemv_max_m else "cublas"

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        x2 = x.reshape(-1, x.shape[-1])
        route = self.route(x2.shape[0])
        if route == "empty":
            return x2.new_empty(*x.shape[:-1], self.out_features)
        if route == "gemv":
            out = fp4gemv.bf16_gemv(x2, self.weight, pdl=self.pdl)
        else:
            out = torch.nn.functional.linear(x2, self.weight)
        return out.view(*x.shape[:-1], self.out_features)

    def gate_up_silu_mul(self, x: torch.Tensor) -> torch.Tensor | None:
        if x.dim() != 2 or self.out_features % 32 != 0 or self.route(x.shape[0]) != "gemv":
            return None
        return fp4gemv.bf16_gemv(x, self.weight, silu_mul=True, pdl=self.pdl)


class NvFp4W4A4Linear(torch.nn.Module):
    """y = bf16(fp32(quant(x) @ dequant(W)^T) * alpha): the W4A4 linear of the
    flashinfer page's NVFP4 kernels (apply_weights: scaled_fp4_quant(x,
    input_global_scale_inv), then the NVFP4 GEMM with alpha).

    weight / weight_scale as for ``NvFp4Linear`` (flat, unpadded scales);
    input_global_scale_inv and alpha: fp32 [1] on the weight's device (alpha
    = the activation's 1 / input_global_scale_inv times the weight's global
    scale).  Up to ``MAX_M`` tokens the library's W4A4 call; beyond, the
    quantiser's exactly dequantised activations and the dequantized weight on
    cuBLAS with alpha applied to the fp32 accumulator (the same products, so
    the same numbers up to the order of the fp32 sums).  ``last_codes``
    holds the latest call's NVFP4 activations (codes, scales)."""

    def __init__(self, weight: torch.Tensor, weight_scale: torch.Tensor, input_global_scale_inv: torch.Tensor,
                 alpha: torch.Tensor, pdl: bool = True):
        super().__init__()
        if weight.dtype != torch.uint8 or weight.dim() != 2 or not weight.is_contiguous():
            raise ValueError("weight must be a contiguous uint8 [N, K/2] tensor")
        N, K = weight.shape[0], weight.shape[1] * 2
        sf = fp4gemv.flat_scale_buffer(weight_scale)
        if sf.numel() < fp4gemv.scale_bytes(N, K):
            raise ValueError(f"weight_scale must hold at least {fp4gemv.scale_bytes(N, K)} bytes")
        for name, t in (("input_global_scale_inv", input_global_scale_inv), ("alpha", alpha)):
            if t.dtype != torch.float32 or t.numel() != 1:
                raise ValueError(f"{name} must be one float32 value")
        self.register_buffer("weight", weight, persistent=False)
        self.register_buffer("weight_scale", sf, persistent=False)
        self.register_buffer("input_global_scale_inv", input_global_scale_inv.reshape(1), persistent=False)
        self.register_buffer("alpha", alpha.reshape(1), persistent=False)
        self.alpha_host = float(alpha.reshape(()).item())  # alpha of the cuBLAS path
        self.out_features, self.in_features = N, K
        self.pdl = bool(pdl)
        self.last_codes = None

    def route(self, m: int) -> str:
        """'empty', 'w4a4' (the library's call) or 'dequant_gemm' (cuBLAS)."""
        if m == 0:
            return "empty"
        return "w4a4" if m <= MAX_M else "dequant_gemm"

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        x2 = x.reshape(-1, x.shape[-1])
        m, K = x2.shape
        route = self.route(m)
        if route == "empty":
            return x2.new_empty(*x.shape[:-1], self.out_features)
        xq = torch.empty(m, K // 2, dtype=torch.uint8, device=x2.device)
        xsf = torch.empty(fp4gemv.scale_bytes(m, K), dtype=torch.uint8, device=x2.device)
        if route == "w4a4":
            out = fp4gemv.w4a4_linear(x2, self.input_global_scale_inv, self.weight, self.weight_scale, self.alpha,
                                      x_fp4=xq, x_sf=xsf, pdl=self.pdl)
        else:
            xd = torch.empty(m, K, dtype=torch.bfloat16, device=x2.device)
            fp4gemv.quantize_act(x2, self.input_global_scale_inv, x_fp4=xq, x_sf=xsf, x_deq=xd)
            w = fp4gemv.dequantize_rows(self.weight, self.weight_scale)
            out = torch.empty(m, self.out_features, dtype=torch.bfloat16, device=x2.device)
            matmul = torch.backends.cuda.matmul
            prev = matmul.allow_bf16_reduced_precision_reduction
            matmul.allow_bf16_reduced_precision_reduction = False  # fp32 split-K sums
            try:
                torch.addmm(out, xd, w.t(), beta=0, alpha=self.alpha_host, out=out)
            finally:
                matmul.allow_bf16_reduced_precision_reduction = prev
        self.last_codes = (xq, xsf)
        return out.view(*x.shape[:-1], self.out_features)
