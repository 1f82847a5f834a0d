"""The token-count dispatch of the linear layers (moe_nvfp4_gemv_gb300.linear).

CPU: the routing rule and the argument checks.  GPU (marked): every route
against the FP64 oracle -- the GEMV for 1 .. 128 tokens, the library's
dequantize + GEMM from dequant_min_m, cuBLAS past 128 tokens -- on 2-D and
3-D inputs, the fused silu_mul path, and the BF16 layer."""
import numpy as np
import pytest
import torch

import oracle
from moe_nvfp4_gemv_gb300 import linear, synth


def _layer(N=256, K=512, dev="cpu", **kw):
    w = synth.fp4_bytes(N, K, seed=N)
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=N + 1)
    gs = torch.tensor([0.01])
    return linear.NvFp4Linear(w.to(dev), sf.to(dev), gs.to(dev), **kw), w, sf


def test_gemv_tile():
    assert [linear.gemv_tile(m) for m in (0, 1, 8, 9, 16, 17, 32, 33, 64, 65, 128, 129)] == \
        [None, 8, 8, 16, 16, 32, 32, 64, 64, 128, 128, None]


def test_routes():
    lin, _, _ = _layer()
    assert lin.route(0) == "empty"
    assert all(lin.route(m) == "gemv" for m in (1, 8, 32, 128))
    assert lin.route(129) == "dequant_gemm" and lin.route(4096) == "dequant_gemm"
    lin2, _, _ = _layer(dequant_min_m=48)
    assert lin2.route(47) == "gemv" and lin2.route(48) == "dequant_gemm"
    b = linear.Bf16Linear(torch.zeros(64, 128, dtype=torch.bfloat16), gemv_max_m=16)
    assert (b.route(0), b.route(16), b.route(17)) == ("empty", "gemv", "cublas")
    w4 = linear.NvFp4W4A4Linear(synth.fp4_bytes(256, 512, seed=1), synth.e4m3_bytes(oracle.scale_bytes(256, 512),
                                                                                       seed=2),
                                torch.tensor([30.0]), torch.tensor([0.001]))
    assert (w4.route(0), w4.route(1), w4.route(128), w4.route(129)) == ("empty", "w4a4", "w4a4", "dequant_gemm")


def test_argument_checks():
    w = synth.fp4_bytes(256, 512, seed=1)
    sf = synth.e4m3_bytes(oracle.scale_bytes(256, 512), seed=2)
    gs = torch.tensor([0.01])
    with pytest.raises(ValueError):
        linear.NvFp4Linear(w.to(torch.int32), sf, gs)
    with pytest.raises(ValueError):
        linear.NvFp4Linear(w, sf[:-4], gs)
    with pytest.raises(ValueError):
        linear.NvFp4Linear(w, sf, torch.tensor([0.01, 0.02]))
    with pytest.raises(ValueError):
        linear.Bf16Linear(torch.zeros(4, 4))


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 5, 16, 40, 128, 129, 300])
def test_nvfp4_linear_routes_match_oracle(M):
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    N, K = 1024, 768
    lin, w, sf = _layer(N, K, dev="cuda")
    x = synth.activations(M, K, seed=M)
    got = lin(x.cuda())
    rows = np.arange(0, N, 7)
    ref = oracle.nvfp4_gemv(_u16(x), w.numpy(), sf.numpy(), 0.01, rows=rows)
    ok, excess, nbad, _ = oracle.check(_u16(got)[:, rows], ref)
    assert ok, (lin.route(M), nbad, excess)


@pytest.mark.gpu
def test_nvfp4_linear_3d_input_and_empty():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    N, K = 512, 512
    lin, w, sf = _layer(N, K, dev="cuda")
    x = synth.activations(6, K, seed=3)
    got = lin(x.view(2, 3, K).cuda())
    assert got.shape == (2, 3, N)
    ref = oracle.nvfp4_gemv(_u16(x), w.numpy(), sf.numpy(), 0.01)
    assert oracle.check(_u16(got.reshape(6, N)), ref)[0]
    assert lin(torch.empty(0, K, dtype=torch.bfloat16, device="cuda")).shape == (0, N)


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 12, 200])
def test_gate_up_silu_mul(M):
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    N, K = 1024, 512
    lin, w, sf = _layer(N, K, dev="cuda")
    x = synth.activations(M, K, seed=M + 9)
    got = lin.gate_up_silu_mul(x.cuda())
    if M > linear.MAX_M:
        assert got is None
        return
    ref = oracle.nvfp4_gemv(_u16(x), w.numpy(), sf.numpy(), 0.01, silu_mul=True)
    assert oracle.check(_u16(got), ref)[0]


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 8, 64, 200])
def test_bf16_linear(M):
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    N, K = 512, 768
    wb = synth.bf16_weight(N, K, seed=5)
    lin = linear.Bf16Linear(wb.cuda())
    x = synth.activations(M, K, seed=M)
    got = lin(x.cuda())
    ref = oracle.bf16_gemv(_u16(x), _u16(wb))
    assert oracle.check(_u16(got), ref)[0], lin.route(M)


# --- scale buffers held by another library: strided views, padding along K --------------

def _padded_scales(sf_exact: torch.Tensor, N: int, K: int, kb_pad: int, fill: int = 0x7F) -> torch.Tensor:
    """The same scales in a buffer whose 128-row groups hold kb_pad 16-wide K
    blocks; the extra 512-byte chunks of each group are filled with `fill`
    (0x7F = NaN in E4M3, so a read of the padding would show)."""
    kbp = (K // 16 + 3) // 4 * 4
    groups = (N + 127) // 128
    src = sf_exact.view(groups, kbp // 4, 512)
    out = torch.full((groups, kb_pad // 4, 512), fill, dtype=torch.uint8)
    out[:, : kbp // 4] = src
    return out.reshape(-1)


def test_flat_scale_buffer_of_a_strided_view():
    from moe_nvfp4_gemv_gb300 import fp4gemv
    N, K = 256, 512
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=4)
    view = sf.view(torch.float8_e4m3fn).view(N // 128, K // 64, 32, 4, 4).permute(0, 2, 3, 1, 4)
    assert not view.is_contiguous()
    flat = fp4gemv.flat_scale_buffer(view)
    assert flat.dtype == torch.uint8 and flat.data_ptr() == sf.data_ptr() and torch.equal(flat, sf)
    with pytest.raises(ValueError):
        fp4gemv.flat_scale_buffer(view[1:])  # does not start the storage


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,silu", [(1, 512, 1024, False), (6, 1056, 768, True), (13, 256, 512, False),
                                        (40, 384, 1280, False), (1, 28672, 4096, True)])
def test_padded_and_strided_scales_match_exact(M, N, K, silu):
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from moe_nvfp4_gemv_gb300 import fp4gemv
    w = synth.fp4_bytes(N, K, seed=N + K)
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=N + K + 1)
    x = synth.activations(M, K, seed=M)
    gs = torch.tensor([0.01], device="cuda")
    xd, wd = x.cuda(), w.cuda()
    exact = fp4gemv.nvfp4_gemv(xd, wd, sf.cuda(), gs, silu_mul=silu)
    kb_pad = (K // 16 + 3) // 4 * 4 + 8
    padded = fp4gemv.nvfp4_gemv(xd, wd, _padded_scales(sf, N, K, kb_pad).cuda(), gs, silu_mul=silu,
                                sf_k_blocks=kb_pad)
    groups = (N + 127) // 128
    view = sf.cuda().view(torch.float8_e4m3fn).view(groups, (K // 16 + 3) // 4, 32, 4, 4).permute(0, 2, 3, 1, 4)
    strided = fp4gemv.nvfp4_gemv(xd, wd, view, gs, silu_mul=silu)
    torch.cuda.synchronize()
    assert torch.equal(padded, exact) and torch.equal(strided, exact)
    if N <= 2048:
        ref = oracle.nvfp4_gemv(_u16(x), w.numpy(), sf.numpy(), 0.01, silu_mul=silu)
        assert oracle.check(_u16(exact), ref)[0]


@pytest.mark.gpu
def test_padded_scales_dequantize_rows_and_linear():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from moe_nvfp4_gemv_gb300 import fp4gemv
    N, K = 384, 1024
    w = synth.fp4_bytes(N, K, seed=8)
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=9)
    kb_pad = K // 16 + 12
    sfp = _padded_scales(sf, N, K, kb_pad).cuda()
    got = fp4gemv.dequantize_rows(w.cuda(), sfp, sf_k_blocks=kb_pad)
    torch.cuda.synchronize()
    assert np.array_equal(_u16(got), oracle.dequantize_rows(w.numpy(), sf.numpy()))
    lin = linear.NvFp4Linear(w.cuda(), sfp, torch.tensor([0.01], device="cuda"), sf_k_blocks=kb_pad)
    for M in (3, 150):  # the GEMV, then dequantize + cuBLAS
        x = synth.activations(M, K, seed=M)
        ref = oracle.nvfp4_gemv(_u16(x), w.numpy(), sf.numpy(), 0.01)
        assert oracle.check(_u16(lin(x.cuda())), ref)[0], M


@pytest.mark.gpu
@pytest.mark.parametrize("M", [3, 128, 300])
def test_w4a4_linear_routes_match_oracle(M):
    # the library's W4A4 call up to 128 tokens, cuBLAS on the dequantised
    # operands beyond: both against the oracle's quantiser and GEMM
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    N, K = 384, 1024
    w = synth.fp4_bytes(N, K, seed=5)
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=6)
    gsi, wgs = 448.0 * 6 / 5.0, 0.02
    alpha = float(np.float32(wgs / gsi))
    lin = linear.NvFp4W4A4Linear(w.cuda(), sf.cuda(), torch.tensor([gsi]).cuda(), torch.tensor([alpha]).cuda())
    x = synth.activations(M, K, seed=M)
    y = lin(x.cuda())
    xq, xsf = oracle.quantize_act(_u16(x), gsi)
    assert np.array_equal(lin.last_codes[0].cpu().numpy(), xq)
    assert np.array_equal(lin.last_codes[1].cpu().numpy(), xsf)
    ok, excess, nbad, _ = oracle.check(_u16(y), oracle.w4a4_gemm(xq, xsf, w.numpy(), sf.numpy(), alpha))
    assert ok, f"{lin.route(M)} M={M}: {nbad} outside tolerance (excess {excess})"
