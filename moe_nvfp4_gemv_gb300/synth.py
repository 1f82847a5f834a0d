"""Seeded synthetic inputs shared by the tests, the bench and the smoke run.

This module holds NO arithmetic of the method: no decoding, no scale layout,
no contraction.  It only draws random numbers of the shapes and value
distributions of the workloads:

* activations ``x``: bf16 ~ N(0, 1) (and a wide-range variant with a few
  entries of very large or very small magnitude);
* NVFP4 weights: uint8 bytes uniform on 0..255 (two uniform 4-bit codes);
* block scales: every byte of the flat scale buffer is float8_e4m3fn(2^U),
  U ~ Uniform[-3, 3] (round-to-nearest cast).  Because each logical scale
  occupies one byte of the buffer, filling the whole buffer i.i.d. gives the
  same distribution under any layout -- callers pass the buffer size, which
  they take from the library (``fp4gemv_scale_bytes``) or the oracle;
* BF16 weights: bf16 ~ N(0, 8^2) (8 is the rms of e2m1 * e4m3(2^U) under the
  distributions above: sqrt(8.5625 * 7.69));
* MoE routing: logits ~ N(0, 1) of shape [M, E]; ids = top-k (no repeats);
  tw = fp32 softmax over the selected logits; alpha[e] = alpha2[e] =
  0.01 * (1 + e / 256); gssh = gssd = 0.01.

All draws use an explicit ``torch.Generator`` seeded per tensor, on the
requested device (CPU draws and CUDA draws of the same seed differ; parity
tests draw on the CPU and copy the same bytes to the GPU).
"""
from __future__ import annotations

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def activations(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """bf16 [M, K] ~ N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn(M, K, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def activations_wide_range(M: int, K: int, seed: int, device="cpu", frac: float = 0.01) -> torch.Tensor:
    """bf16 [M, K] ~ N(0, 1) where a fraction `frac` of the entries in the
    first half of K is replaced by a value of the same sign and magnitude
    10^V, V ~ Uniform[5, 7] or Uniform[-9, -6] with equal odds (far outside
    the f16 range, or below its subnormal grid).  The second half of K keeps
    the plain N(0, 1) draw."""
    g = _gen(seed, device)
    x = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    pick = torch.rand(M, K, generator=g, device=device) < frac
    pick[:, K // 2:] = False
    big = torch.rand(M, K, generator=g, device=device) < 0.5
    v = torch.rand(M, K, generator=g, device=device)
    mag = torch.where(big, torch.pow(10.0, 5.0 + 2.0 * v), torch.pow(10.0, -9.0 + 3.0 * v))
    x = torch.where(pick, torch.sign(x) * mag, x)
    return x.to(torch.bfloat16)


def fp4_bytes(rows: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """uint8 [rows, K/2], every byte uniform on 0..255."""
    g = _gen(seed, device)
    return torch.randint(0, 256, (rows, K // 2), generator=g, device=device, dtype=torch.int32).to(torch.uint8)


def e4m3_bytes(nbytes: int, seed: int, device="cpu", lo: float = -3.0, hi: float = 3.0) -> torch.Tensor:
    """uint8 [nbytes], each byte float8_e4m3fn(2^U), U ~ Uniform[lo, hi]."""
    g = _gen(seed, device)
    u = torch.rand(nbytes, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo
    return torch.exp2(u).to(torch.float8_e4m3fn).view(torch.uint8)


def bf16_weight(rows: int, K: int, seed: int, device="cpu", std: float = 8.0) -> torch.Tensor:
    """bf16 [rows, K] ~ N(0, std^2)."""
    g = _gen(seed, device)
    return (torch.randn(rows, K, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def routing(M: int, E: int, topk: int, seed: int, device="cpu"):
    """(ids int32 [M, topk], tw fp32 [M, topk]): top-k of N(0,1) logits and
    the fp32 softmax of the selected logits."""
    g = _gen(seed, device)
    logits = torch.randn(M, E, generator=g, device=device, dtype=torch.float32)
    vals, ids = torch.topk(logits, topk, dim=1)
    tw = torch.softmax(vals, dim=1)
    return ids.to(torch.int32).contiguous(), tw.to(torch.float32).contiguous()


def expert_alphas(E: int, device="cpu") -> torch.Tensor:
    """fp32 [E]: 0.01 * (1 + e / 256), distinct per expert."""
    e = torch.arange(E, device=device, dtype=torch.float32)
    return (0.01 * (1.0 + e / 256.0)).to(torch.float32)


# Workload shapes (the configurations the tests and the bench use).
TINY = dict(M=1, N=256, K=512, gs=0.01)
LLAMA8B_LAYERS = {  # (N, K, silu_mul)
    "qkv": (6144, 4096, False),
    "o_proj": (4096, 4096, False),
    "gate_up": (28672, 4096, True),
    "down": (4096, 14336, False),
}
LLAMA8B_M = (1, 2, 4, 8, 16, 32)
LLAMA70B_LAYERS = {
    "gate_up": (57344, 8192, True),
    "down": (8192, 28672, False),
    "qkv": (10240, 8192, False),
}
LLAMA70B_M = (1, 4, 16, 32)
MOE = dict(E=128, H=4096, I=1536, SI=1536, topk=8)
MOE_M = (1, 8, 32)
SWEEP_NK = 8192
SWEEP_M = (1, 2, 4, 8, 16, 24, 32, 48, 64, 96, 128)
