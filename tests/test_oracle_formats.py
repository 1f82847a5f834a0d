"""Pins for the oracle's number formats and scale layout (CPU only).

Each test checks the oracle against something other than itself: the value
table the pages imply, torch's float8_e4m3fn / bfloat16 conversions (library
routines), exhaustive invariants, the pages' buffer-size formula.
"""
import math
import struct

import numpy as np
import pytest
import torch

import oracle


# E2M1 magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6} with the sign in bit 3: the FP4
# value set of NVFP4 (vllm.models.flint.ops.nvfp4_gemv, module docstring,
# "E2M1 codes").
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_table():
    for code, want in enumerate(E2M1_TABLE):
        got = oracle.e2m1(code)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), code


def test_e4m3_all_256_codes_match_torch():
    # torch's float8_e4m3fn -> float32 conversion is an independent library routine.
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)
    for b in range(256):
        got, want = oracle.e4m3(b), float(ref[b])
        if math.isnan(want):
            assert math.isnan(got), b
        else:
            assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), (b, got, want)
    assert oracle.e4m3(0x7E) == 448.0 and oracle.e4m3(0x01) == 2.0 ** -9


def test_dequant_products_are_exact_in_bf16():
    # "every weight is dequantized exactly to BF16": all 16 x 256 (code, scale)
    # products with a finite scale round-trip through bf16 unchanged.
    for b in range(256):
        s = oracle.e4m3(b)
        if math.isnan(s):
            continue
        for code in range(16):
            p = oracle.e2m1(code) * s
            assert oracle.bf16_value(oracle.bf16_rne(p)) == p, (code, b)


def _f32_bits_to_bf16_torch(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    return [int(v) & 0xFFFF for v in t.view(torch.int16).tolist()]


def test_bf16_rne_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    # ties, subnormals, near-overflow and zero
    extra = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 2.0 ** -130, 2.0 ** -133, 2.0 ** -134,
             3 * 2.0 ** -135, 3.3895313892515355e38, 3.3961775292304e38, 0.0, -0.0, 65504.0]
    vals = np.concatenate([vals, np.array(extra, np.float32)])
    want = _f32_bits_to_bf16_torch(vals.tolist())
    for v, w in zip(vals.tolist(), want):
        assert oracle.bf16_rne(v) == w, (v, hex(w))


def test_bf16_rne_rounds_double_directly():
    # 1 + 2^-8 + 2^-30 lies just above a bf16 tie: one direct rounding gives
    # 1 + 2^-7; rounding through float32 first (which lands on the tie) would
    # give 1.0.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert oracle.bf16_value(oracle.bf16_rne(v)) == 1.0 + 2.0 ** -7
    assert oracle.bf16_value(oracle.bf16_rne(-v)) == -(1.0 + 2.0 ** -7)
    assert oracle.bf16_value(oracle.bf16_rne(1.0 + 2.0 ** -8)) == 1.0  # exact tie -> even
    assert oracle.bf16_rne(float("inf")) == 0x7F80
    assert oracle.bf16_rne(3.4e38) == 0x7F80  # rounds past the largest finite bf16
    assert math.isnan(oracle.bf16_value(oracle.bf16_rne(float("nan"))))


def pages_scale_nbytes(n, k):
    # _swizzled_scale_buffer (vllm.models.flint.ops.linear): the flat 128x4
    # buffer size, as printed on the page.
    return (n + 127) // 128 * 128 * ((k // 16 + 3) // 4 * 4)


@pytest.mark.parametrize("rows,K", [(256, 512), (16, 32), (130, 80), (1, 16), (384, 4096), (3072, 1536)])
def test_scale_layout_bijection_and_size(rows, K):
    nbytes = oracle.scale_bytes(rows, K)
    assert nbytes == pages_scale_nbytes(rows, K)
    rp = (rows + 127) // 128 * 128
    kbp = (K // 16 + 3) // 4 * 4
    seen = np.zeros(nbytes, np.int32)
    for r in range(rp):
        for kb in range(kbp):
            off = oracle.swz(r, kb, K)
            assert 0 <= off < nbytes
            seen[off] += 1
            assert oracle.unswz(off, K) == (r, kb)
    assert (seen == 1).all()


def test_scale_layout_chunk_structure():
    # Structure of the reading of the 128x4 layout: each 128-row x 4-block tile
    # occupies one 512-byte aligned chunk, the 4 K blocks of a row are
    # adjacent bytes, and chunks advance along K first within a 128-row group.
    K = 1024  # 64 blocks -> 16 chunks per 128-row group
    for r in (0, 5, 31, 32, 77, 127, 128, 300):
        for kb in (0, 3, 4, 17, 63):
            off = oracle.swz(r, kb, K)
            assert off // 512 == (r // 128) * 16 + kb // 4
            assert oracle.swz(r, kb - kb % 4, K) + kb % 4 == off
    base = {oracle.swz(r, kb, K) // 512 for r in range(128) for kb in range(4)}
    assert base == {0}
