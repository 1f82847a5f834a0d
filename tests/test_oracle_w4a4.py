"""Pins for the oracle's W4A4 pieces (CPU only): the E2M1 / E4M3 encoders,
the activation quantiser and the NVFP4 x NVFP4 GEMM
(vllm.model_executor.kernels.linear.nvfp4.flashinfer, the W4A4 kernels'
apply_weights: scaled_fp4_quant, then the NVFP4 GEMM with alpha).

The pages do not print the quantiser's arithmetic; the oracle states its
reading.  These tests check the oracle against things other than itself:
the E2M1 value set, torch's float8_e4m3fn conversion (a library routine),
nearest-value and tie properties checked over every grid point, hand-worked
blocks (tests/golden/w4a4_quant_block.json), lossless and scaling
invariants, and the dense GEMV oracle on activations that quantise exactly.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
HERE = os.path.dirname(os.path.abspath(__file__))


def bf16_bits(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_e2m1_encode_round_trip():
    for c in range(16):
        assert oracle.e2m1_encode(oracle.e2m1(c)) == (0 if c == 8 else c), c


def test_e2m1_encode_nearest_and_ties():
    # every value on a fine grid maps to a nearest E2M1 magnitude; exact ties
    # take the even code; beyond 6 saturates; the sign follows v unless zero
    grid = np.arange(-8.0, 8.0 + 1e-9, 1.0 / 64).astype(np.float32)
    for v in grid.tolist():
        c = oracle.e2m1_encode(v)
        mag = E2M1_MAG[c & 7]
        d = abs(abs(v) - mag)
        assert all(d <= abs(abs(v) - m) for m in E2M1_MAG), (v, c)
        ties = [i for i, m in enumerate(E2M1_MAG) if abs(abs(v) - m) == d]
        if len(ties) > 1:
            assert (c & 7) % 2 == 0, (v, c)
        assert (c & 8) == (8 if (v < 0 and (c & 7) != 0) else 0), (v, c)
    # the midpoints, by hand: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    assert [oracle.e2m1_encode(v) for v in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)] == [0, 2, 2, 4, 4, 6, 6]
    assert oracle.e2m1_encode(1e30) == 7 and oracle.e2m1_encode(-1e30) == 15 and oracle.e2m1_encode(-0.2) == 0


def test_e4m3_encode_round_trip():
    for c in range(0x7F):
        assert oracle.e4m3_encode(oracle.e4m3(c)) == c, c


def test_e4m3_encode_matches_torch():
    # torch's float32 -> float8_e4m3fn conversion rounds to nearest even
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.uniform(0, 448, 4000), np.exp2(rng.uniform(-12, 8.8, 4000))]).astype(np.float32)
    v = v[v <= 448.0]
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(a)) for a in v], np.uint8)
    assert np.array_equal(got, want)
    # saturation (finite): above 448 -> 448
    assert oracle.e4m3_encode(449.0) == 0x7E and oracle.e4m3_encode(1e9) == 0x7E


def test_quantize_golden_blocks():
    cases = json.load(open(os.path.join(HERE, "golden", "w4a4_quant_block.json")))["cases"]
    for c in cases:
        q, sf = oracle.quantize_act(bf16_bits(c["x"]).reshape(1, 16), c["gsi"])
        assert q[0].tolist() == c["bytes"], c["name"]
        assert int(sf[oracle.swz(0, 0, 16)]) == c["scale"], c["name"]


def _lossless_x(M, K, seed):
    """Activations that quantise exactly under gsi = 1: each block holds E2M1
    magnitudes times 2^e with one element at 6 * 2^e (so s = 2^e, an exact
    E4M3 power of two, and x * r lands on the grid)."""
    rng = np.random.default_rng(seed)
    x = np.empty((M, K), np.float32)
    for m in range(M):
        for b in range(K // 16):
            e = int(rng.integers(-6, 6))
            vals = np.array(E2M1_MAG, np.float32)[rng.integers(0, 8, 16)] * rng.choice([-1.0, 1.0], 16)
            vals[rng.integers(0, 16)] = 6.0 * rng.choice([-1.0, 1.0])
            x[m, 16 * b:16 * b + 16] = vals * np.float32(2.0 ** e)
    x[x == 0] = 0.0  # (+0: a zero is stored as code 0)
    return bf16_bits(x.reshape(-1)).reshape(M, K)


def test_quantize_lossless_round_trip():
    M, K = 5, 256
    x = _lossless_x(M, K, 1)
    q, sf = oracle.quantize_act(x, 1.0)
    assert np.array_equal(oracle.dequantize_rows(q, sf), x)
    # padding rows and blocks of the 128x4 buffer stay zero
    used = {oracle.swz(m, b, K) for m in range(M) for b in range(K // 16)}
    assert all(sf[i] == 0 for i in range(sf.size) if i not in used)


def test_quantize_scaling_invariants():
    rng = np.random.default_rng(2)
    x = bf16_bits(rng.standard_normal(8 * 128).astype(np.float32)).reshape(8, 128)
    q, sf = oracle.quantize_act(x, 37.0)
    # doubling x (exact in bf16) doubles every scale and keeps the codes,
    # while no scale saturates
    x2 = bf16_bits((torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float() * 2).reshape(-1).tolist())
    q2, sf2 = oracle.quantize_act(x2.reshape(8, 128), 37.0)
    assert np.array_equal(q, q2)
    used = [oracle.swz(m, b, 128) for m in range(8) for b in range(8)]
    for i in used:
        assert oracle.e4m3(int(sf2[i])) == 2 * oracle.e4m3(int(sf[i]))
    # gsi scales the stored scales the same way (and the codes not at all)
    q3, sf3 = oracle.quantize_act(x, 74.0)
    assert np.array_equal(q, q3)
    for i in used:
        assert oracle.e4m3(int(sf3[i])) == 2 * oracle.e4m3(int(sf[i]))
    # each element is within half the local E2M1 spacing of x * r
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy()
    for m in range(8):
        for b in range(8):
            s = oracle.e4m3(int(sf[oracle.swz(m, b, 128)]))
            for i in range(16):
                k = 16 * b + i
                c = (q[m, k // 2] >> (4 * (k % 2))) & 0xF
                v = float(np.float32(xf[m, k]) * np.float32(np.float32(37.0) / np.float32(s)))
                got = oracle.e2m1(c)
                assert min(abs(v - g) for g in E2M1_MAG + [-g for g in E2M1_MAG]) == abs(v - got) or abs(v) > 6


@pytest.mark.parametrize("M,N,K", [(3, 64, 256), (9, 48, 512)])
def test_w4a4_gemm_equals_w4a16_on_lossless_activations(M, N, K):
    # activations that quantise exactly: the W4A4 GEMM with alpha = gs / gsi
    # is the dense NVFP4 GEMV of the original activations
    from moe_nvfp4_gemv_gb300 import synth
    x = _lossless_x(M, K, 7)
    w = synth.fp4_bytes(N, K, seed=5).numpy()
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=6).numpy()
    gsi, gs = 4.0, 0.01
    xs = bf16_bits((torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float() / gsi).reshape(-1).tolist())
    q, xsf = oracle.quantize_act(xs.reshape(M, K), gsi)
    got = oracle.w4a4_gemm(q, xsf, w, sf, gs / gsi)
    want = oracle.nvfp4_gemv(xs.reshape(M, K), w, sf, gs)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)
