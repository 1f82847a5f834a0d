"""The W4A4 path on the GPU against the oracle
(vllm.model_executor.kernels.linear.nvfp4.flashinfer, the W4A4 kernels'
apply_weights: scaled_fp4_quant, then the NVFP4 x NVFP4 GEMM with alpha).

The quantiser's codes and scales are integer results decided in binary32 on
both sides, so they must match bit for bit, padding bytes of the 128x4
layout included.  The GEMM output goes through the per-element tolerance
rule, as every GEMV output does.  Shapes span several 128-row scale groups,
a ragged last group, K-block padding (K / 16 not a multiple of 4), and GEMMs
of more than 128 rows (several launches)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, require_gpu, sample_rows, u16
from moe_nvfp4_gemv_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def fp4():
    require_gpu()
    from moe_nvfp4_gemv_gb300 import fp4gemv
    return fp4gemv


def act_inputs(M, K, seed, kind):
    """bf16 activations: normal; log-uniform magnitudes over 2^-30 .. 2^10
    with random signs (many blocks with tiny scales, some subnormal E4M3);
    or normal with some all-zero blocks and exact zeros."""
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        x = torch.randn(M, K, generator=g)
    elif kind == "wide":
        x = torch.exp2(torch.rand(M, K, generator=g) * 40 - 30) * (torch.randint(0, 2, (M, K), generator=g) * 2 - 1)
    else:
        x = torch.randn(M, K, generator=g)
        x[torch.rand(M, K, generator=g) < 0.2] = 0.0
        blocks = x.view(M, K // 16, 16)
        blocks[torch.rand(M, K // 16, generator=g) < 0.1] = 0.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("M,K,kind,gsi", [(1, 256, "normal", 1.0), (5, 272, "wide", 37.0),
                                          (130, 512, "zeros", 448.0 * 6 / 4.5), (128, 4096, "normal", 2.0 ** -3),
                                          (3, 64, "wide", 2.0 ** 20)])
def test_quantize_act_bit_exact(fp4, M, K, kind, gsi):
    x = act_inputs(M, K, seed=M + K, kind=kind)
    gs = torch.tensor([gsi], dtype=torch.float32, device=DEV)
    q = torch.full((M, K // 2), 0xA5, dtype=torch.uint8, device=DEV)
    sf = torch.full((fp4.scale_bytes(M, K),), 0xA5, dtype=torch.uint8, device=DEV)
    fp4.quantize_act(x.to(DEV), gs, x_fp4=q, x_sf=sf)
    rq, rsf = oracle.quantize_act(u16(x), gsi)
    assert np.array_equal(q.cpu().numpy(), rq), "codes"
    assert np.array_equal(sf.cpu().numpy(), rsf), "scales (padding included)"
    assert fp4.get_device_error() == 0


def test_quantize_act_strided_rows(fp4):
    # x as a column slice of a wider buffer (row stride > K)
    M, K = 7, 512
    base = act_inputs(M, 1024, seed=9, kind="normal")
    x = base[:, 256:256 + K]
    gs = torch.tensor([3.0], device=DEV)
    q, sf = fp4.quantize_act(base.to(DEV)[:, 256:256 + K], gs)
    rq, rsf = oracle.quantize_act(u16(x), 3.0)
    assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(sf.cpu().numpy(), rsf)


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (8, 384, 1024), (33, 256, 768), (200, 128, 512)])
def test_w4a4_gemm(fp4, M, N, K):
    x = act_inputs(M, K, seed=100 + M, kind="normal")
    w = synth.fp4_bytes(N, K, seed=M + 1)
    wsf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=M + 2)
    gsi, wgs = 448.0 * 6 / 5.0, 0.02
    alpha = wgs / gsi
    xq, xsf = oracle.quantize_act(u16(x), gsi)
    ref = oracle.w4a4_gemm(xq, xsf, w.numpy(), wsf.numpy(), float(np.float32(alpha)))
    at = torch.tensor([alpha], dtype=torch.float32, device=DEV)
    out = fp4.w4a4_gemm(torch.from_numpy(xq).to(DEV), torch.from_numpy(xsf).to(DEV), w.to(DEV), wsf.to(DEV), at)
    assert_close(u16(out), ref, f"w4a4_gemm M={M} N={N} K={K}")
    # the one-call form: the same codes, scales and output
    q, sf = torch.empty_like(torch.from_numpy(xq)).to(DEV), torch.empty(xsf.size, dtype=torch.uint8, device=DEV)
    out2 = fp4.w4a4_linear(x.to(DEV), torch.tensor([gsi], device=DEV), w.to(DEV), wsf.to(DEV), at, x_fp4=q, x_sf=sf)
    assert np.array_equal(q.cpu().numpy(), xq) and np.array_equal(sf.cpu().numpy(), xsf)
    assert torch.equal(out, out2)
    assert fp4.get_device_error() == 0


def test_w4a4_linear_llama8b_gate_up_sampled(fp4):
    # Llama-3-8B gate_up (28672 x 4096) at 128 tokens, sampled output rows
    M, N, K = 128, 28672, 4096
    x = act_inputs(M, K, seed=7, kind="normal")
    w = synth.fp4_bytes(N, K, seed=11)
    wsf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=12)
    gsi, wgs = 448.0 * 6 / 4.0, 0.01
    alpha = float(np.float32(wgs / gsi))
    out = fp4.w4a4_linear(x.to(DEV), torch.tensor([gsi], device=DEV), w.to(DEV), wsf.to(DEV),
                          torch.tensor([alpha], device=DEV))
    rows = sample_rows(N, 48, seed=3)
    xq, xsf = oracle.quantize_act(u16(x), gsi)
    ref = oracle.w4a4_gemm(xq, xsf, w.numpy(), wsf.numpy(), alpha, rows=rows)
    assert_close(u16(out)[:, rows], ref, "w4a4 gate_up M=128 (sampled rows)")
    assert fp4.get_device_error() == 0


def _random_shapes():
    rng = np.random.default_rng(44)
    return [(int(rng.integers(1, 301)), 16 * int(rng.integers(1, 65)), 64 * int(rng.integers(4, 33))) for _ in range(8)]


@pytest.mark.parametrize("M,N,K", _random_shapes())
def test_w4a4_random_shapes(fp4, M, N, K):
    # seeded random shapes: codes and scales bit-exact, outputs (sampled rows
    # past 256 features) under the tolerance, through w4a4_linear
    x = act_inputs(M, K, seed=M * 7 + K, kind="wide" if M % 2 else "normal")
    w = synth.fp4_bytes(N, K, seed=N + K)
    wsf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=N + K + 1)
    gsi = float(2.0 ** (M % 7 - 2))
    alpha = float(np.float32(0.01 / gsi))
    q = torch.empty(M, K // 2, dtype=torch.uint8, device=DEV)
    sf = torch.empty(oracle.scale_bytes(M, K), dtype=torch.uint8, device=DEV)
    out = fp4.w4a4_linear(x.to(DEV), torch.tensor([gsi], device=DEV), w.to(DEV), wsf.to(DEV),
                          torch.tensor([alpha], device=DEV), x_fp4=q, x_sf=sf)
    xq, xsf = oracle.quantize_act(u16(x), gsi)
    assert np.array_equal(q.cpu().numpy(), xq) and np.array_equal(sf.cpu().numpy(), xsf)
    rows = None if N <= 256 else sample_rows(N, 40, seed=M)
    ref = oracle.w4a4_gemm(xq, xsf, w.numpy(), wsf.numpy(), alpha, rows=rows)
    got = u16(out) if rows is None else u16(out)[:, rows]
    assert_close(got, ref, f"w4a4 random M={M} N={N} K={K}")
    assert fp4.get_device_error() == 0


def test_w4a4_linear_chained_under_pdl(fp4):
    # w4a4_linear right after the GEMV that writes its input, both with PDL:
    # the quantisation (launched early) must wait for that GEMV's outputs.
    # Chained results equal the same calls run one by one, bit for bit.
    M, K, N = 4, 1024, 512
    x = act_inputs(M, K, seed=3, kind="normal").to(DEV)
    w1 = synth.fp4_bytes(K, K, seed=21).to(DEV)
    s1 = synth.e4m3_bytes(oracle.scale_bytes(K, K), seed=22).to(DEV)
    w2 = synth.fp4_bytes(N, K, seed=23).to(DEV)
    s2 = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=24).to(DEV)
    gs = torch.tensor([0.05], device=DEV)
    gsi = torch.tensor([448.0 * 6 / 8.0], device=DEV)
    alpha = torch.tensor([0.02 / (448.0 * 6 / 8.0)], device=DEV)
    h_iso = fp4.nvfp4_gemv(x, w1, s1, gs, pdl=False)
    torch.cuda.synchronize()
    y_iso = fp4.w4a4_linear(h_iso, gsi, w2, s2, alpha, pdl=False)
    torch.cuda.synchronize()
    for _ in range(3):
        h = torch.full((M, K), 9.0, dtype=torch.bfloat16, device=DEV)
        fp4.nvfp4_gemv(x, w1, s1, gs, out=h, pdl=True)
        y = fp4.w4a4_linear(h, gsi, w2, s2, alpha, pdl=True)
        torch.cuda.synchronize()
        assert torch.equal(h, h_iso) and torch.equal(y, y_iso)
    assert fp4.get_device_error() == 0
