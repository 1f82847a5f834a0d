"""Pins for the oracle's dense ops (CPU only): hand-worked golden cases,
brute force against an independent decode, a library cross-check against
torch.matmul in float64, closed forms and structural identities."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from moe_nvfp4_gemv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")
E2M1_TABLE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def bf16_bits(vals) -> np.ndarray:
    t = torch.as_tensor(np.asarray(vals, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def place_scales(logical: np.ndarray, K: int) -> np.ndarray:
    rows = logical.shape[0]
    buf = np.zeros(oracle.scale_bytes(rows, K), np.uint8)
    for r in range(rows):
        for kb in range(K // 16):
            buf[oracle.swz(r, kb, K)] = logical[r, kb]
    return buf


def independent_decode(w: np.ndarray, sf_logical: np.ndarray) -> np.ndarray:
    """Decode [N, K/2] codes (low nibble first) with the literal E2M1 table and
    torch's float8_e4m3fn conversion of the logical scales; float64."""
    lo = (w & 0xF).astype(np.int64)
    hi = (w >> 4).astype(np.int64)
    codes = np.stack([lo, hi], axis=-1).reshape(w.shape[0], -1)
    vals = E2M1_TABLE[codes]
    s = torch.as_tensor(sf_logical).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals * np.repeat(s, 16, axis=1)


def finish(acc: np.ndarray, gs: float) -> np.ndarray:
    """bf16(f32(f32(acc) * gs)) using numpy float32 and torch's f32->bf16."""
    v = (acc.astype(np.float32) * np.float32(gs)).astype(np.float32)
    return bf16_bits(v)


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _golden_inputs(c):
    K = c["K"]
    w = np.stack([np.frombuffer(bytes.fromhex(h), np.uint8) for h in c["w_hex"]])
    sf = place_scales(np.array(c["scales"], np.uint8), K)
    x = bf16_bits(np.array(c["x"], np.float32))
    return w, sf, x


def test_golden_dequant(golden):
    for c in golden:
        if "dequant" not in c:
            continue
        w, sf, _ = _golden_inputs(c)
        got = oracle.dequantize_rows(w, sf)
        assert np.array_equal(got, bf16_bits(np.array(c["dequant"], np.float32))), c["name"]


def test_golden_gemv(golden):
    for c in golden:
        w, sf, x = _golden_inputs(c)
        nom, lo, hi = oracle.nvfp4_gemv(x, w, sf, c["gs"], silu_mul=c.get("silu_mul", False))
        assert nom.tolist() == c["out_bits"], c["name"]
        assert np.array_equal(lo, nom) and np.array_equal(hi, nom), c["name"]


@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("gs", [1.0, 0.01])
def test_brute_force_n16_k32(M, gs):
    N, K = 16, 32
    w = synth.fp4_bytes(N, K, seed=11).numpy()
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=12).numpy()
    x = synth.activations(M, K, seed=13).view(torch.int16).numpy().view(np.uint16)
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    wd = independent_decode(w, oracle.scales_logical(sf, N, K))
    acc = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += xd[m, k] * wd[n, k]
            acc[m, n] = s
    nom, _, _ = oracle.nvfp4_gemv(x, w, sf, gs)
    assert np.array_equal(nom, finish(acc, gs))
    # dequantize_rows agrees with the independent decode, bit for bit
    assert np.array_equal(oracle.dequantize_rows(w, sf), bf16_bits(wd.astype(np.float32)))


def test_library_crosscheck_matmul_fp64():
    M, N, K, gs = 4, 256, 512, 0.01
    w = synth.fp4_bytes(N, K, seed=1).numpy()
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=2).numpy()
    x = synth.activations(M, K, seed=3)
    wd = independent_decode(w, oracle.scales_logical(sf, N, K))
    acc = torch.matmul(x.to(torch.float64), torch.from_numpy(wd).T).numpy()
    nom, _, _ = oracle.nvfp4_gemv(x.view(torch.int16).numpy().view(np.uint16), w, sf, gs)
    assert np.array_equal(nom, finish(acc, gs))


def test_closed_form_all_ones_code():
    # W = code 2 (1.0) everywhere, scales powers of two: out = gs * sum_k x_k s_k
    # exactly (small integers; every partial sum exact in fp32).
    N, K, gs = 32, 256, 0.5
    w = np.full((N, K // 2), 0x22, np.uint8)
    logical = np.zeros((N, K // 16), np.uint8)
    for n in range(N):
        for kb in range(K // 16):
            logical[n, kb] = 0x38 + 8 * ((n + kb) % 3)  # 1.0, 2.0, 4.0
    sf = place_scales(logical, K)
    xs = (np.arange(2 * K) % 7 - 3).reshape(2, K).astype(np.float32)
    x = bf16_bits(xs)
    nom, _, _ = oracle.nvfp4_gemv(x, w, sf, gs)
    svals = 2.0 ** ((np.arange(N)[:, None] + np.arange(K // 16)[None, :]) % 3)
    want = np.array([[gs * sum(xs[m, k] * svals[n, k // 16] for k in range(K)) for n in range(N)] for m in range(2)])
    assert np.array_equal(nom, bf16_bits(want.astype(np.float32)))


def test_silu_mul_closed_forms():
    # gate rows all zero -> silu(0) * U = 0 exactly; and the golden silu case
    # pins the nonzero path.
    N, K = 64, 64
    w = synth.fp4_bytes(N, K, seed=5).numpy().copy()
    w[: N // 2] = 0
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=6).numpy()
    x = synth.activations(3, K, seed=7).view(torch.int16).numpy().view(np.uint16)
    nom, lo, hi = oracle.nvfp4_gemv(x, w, sf, 0.01, silu_mul=True)
    assert nom.shape == (3, N // 2)
    assert not np.any(nom & 0x7FFF) and not np.any(lo & 0x7FFF) and not np.any(hi & 0x7FFF)


def test_silu_mul_matches_formula_on_gate_up_outputs():
    # out = bf16(silu(G) * U) with G, U the bf16 outputs of the plain GEMV on
    # the gate and up halves (nominal path).
    N, K, gs = 64, 128, 0.02
    w = synth.fp4_bytes(N, K, seed=8).numpy()
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=9).numpy()
    x = synth.activations(2, K, seed=10).view(torch.int16).numpy().view(np.uint16)
    plain, _, _ = oracle.nvfp4_gemv(x, w, sf, gs)
    G = oracle.bf16_to_f64(plain[:, : N // 2])
    U = oracle.bf16_to_f64(plain[:, N // 2:])
    want = [[oracle.bf16_rne(g / (1.0 + math.exp(-g)) * u) for g, u in zip(gr, ur)] for gr, ur in zip(G, U)]
    nom, lo, hi = oracle.nvfp4_gemv(x, w, sf, gs, silu_mul=True)
    assert nom.tolist() == want
    assert (oracle.bf16_to_f64(lo) <= oracle.bf16_to_f64(nom)).all()
    assert (oracle.bf16_to_f64(nom) <= oracle.bf16_to_f64(hi)).all()


def test_bf16_gemv_equals_nvfp4_on_dequantized_weight():
    # bf16_gemv is "the same kernel with a row-major BF16 weight" and global
    # scale 1: on the dequantized weight it must reproduce nvfp4_gemv(gs=1).
    N, K = 128, 256
    w = synth.fp4_bytes(N, K, seed=21).numpy()
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=22).numpy()
    x = synth.activations(5, K, seed=23).view(torch.int16).numpy().view(np.uint16)
    wb = oracle.dequantize_rows(w, sf)
    for silu in (False, True):
        a = oracle.nvfp4_gemv(x, w, sf, 1.0, silu_mul=silu)
        b = oracle.bf16_gemv(x, wb, silu_mul=silu)
        for u, v in zip(a, b):
            assert np.array_equal(u, v)


def test_sampled_rows_match_full():
    N, K = 96, 128
    w = synth.fp4_bytes(N, K, seed=31).numpy()
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=32).numpy()
    x = synth.activations(3, K, seed=33).view(torch.int16).numpy().view(np.uint16)
    rows = np.array([0, 5, 47, 95])
    full = oracle.nvfp4_gemv(x, w, sf, 0.01)
    samp = oracle.nvfp4_gemv(x, w, sf, 0.01, rows=rows)
    for f, s in zip(full, samp):
        assert np.array_equal(f[:, rows], s)
    fs = oracle.nvfp4_gemv(x, w, sf, 0.01, silu_mul=True)
    ss = oracle.nvfp4_gemv(x, w, sf, 0.01, silu_mul=True, rows=np.array([1, 40]))
    for f, s in zip(fs, ss):
        assert np.array_equal(f[:, [1, 40]], s)


def test_check_rule_detects_planted_mistakes():
    # The acceptance rule must reject a transposed operand or a dropped scale.
    N, K = 64, 256
    w = synth.fp4_bytes(N, K, seed=41).numpy()
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=42).numpy()
    x = synth.activations(4, K, seed=43).view(torch.int16).numpy().view(np.uint16)
    ref = oracle.nvfp4_gemv(x, w, sf, 0.01)
    assert oracle.check(ref[0], ref)[0]
    wrong_gs = oracle.nvfp4_gemv(x, w, sf, 0.0125)[0]
    assert not oracle.check(wrong_gs, ref)[0]
    swapped = oracle.nvfp4_gemv(x[::-1].copy(), w, sf, 0.01)[0]
    assert not oracle.check(swapped, ref)[0]
    nibble_swap = ((w >> 4) | (w << 4)).astype(np.uint8)
    assert not oracle.check(oracle.nvfp4_gemv(x, nibble_swap, sf, 0.01)[0], ref)[0]
