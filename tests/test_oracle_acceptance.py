"""Pins for the oracle's acceptance rule (CPU only).

The tolerance is per element: |gpu - ref| <= 2^-7 |ref| + 2^-10 rms(ref).
The pages round the output once (vllm.models.flint.ops.nvfp4_gemv, module
docstring) and name a few intermediate bf16 roundings (the gate / up values
before silu_mul; y_j, y_shared and the top-k sum in down_combine,
vllm.models.flint.ops.moe_gemv module docstring).  Only those intermediates
carry an alternative rounding, and only when the exact value sits next to a
rounding midpoint.  These tests check that:

* the helper that rounds an intermediate offers the other neighbour exactly
  when a midpoint lies within the window;
* outputs without an intermediate rounding have no window at all, so check()
  is exactly the per-element formula for them;
* with intermediates, the window is empty unless an intermediate computed
  independently here lies next to a midpoint;
* mistakes planted in the oracle's inputs at K = 14336 and 28672 (one dropped
  16-wide K block, every scale one E4M3 step off, gate and up rows swapped)
  fail on most outputs;
* the 2^-16 window is wider than the error of an fp32 round-to-nearest
  accumulation of 16-product blocks, emulated here, for values that are not
  small against the output's rms.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from moe_nvfp4_gemv_gb300 import synth

from test_oracle_gemv import bf16_bits, independent_decode

TOL_REL = 2.0 ** -7
TOL_RMS = 2.0 ** -10


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def formula_bad(gpu_bits, nom_bits):
    """The per-element tolerance written out (no interval)."""
    g = oracle.bf16_to_f64(gpu_bits)
    n = oracle.bf16_to_f64(nom_bits)
    rms = math.sqrt(float(np.mean(n * n)))
    return np.abs(g - n) > TOL_REL * np.abs(n) + TOL_RMS * rms


def bf16_midpoint_distance(v: np.ndarray) -> np.ndarray:
    """|v - nearest bf16 rounding midpoint| for normal float64 values v,
    from the binade's quantum (8 significant bits)."""
    a = np.abs(v)
    e = np.floor(np.log2(a))
    q = np.exp2(e - 7)
    mid = (np.floor(a / q) + 0.5) * q
    return np.minimum(np.abs(a - mid), np.abs(a - (mid - q)))


# ------------------------------------------------------------------------------------------
# the intermediate-rounding helper
# ------------------------------------------------------------------------------------------

def test_round_intermediate_grid_points_have_no_alternative():
    vals = [1.0, -1.0, 3.0, 0.0078125, 1.5, -96.0, 2.0 ** -100, 12288.0]
    for v in vals:
        want = int(bf16_bits([v])[0])
        assert oracle.round_intermediate(v, oracle.INTERMEDIATE_REL_WINDOW * abs(v)) == (want, want)


def test_round_intermediate_midpoints():
    # 1 + 2^-8 lies halfway between 1 (even) and 1 + 2^-7; 1 + 3 * 2^-8
    # halfway between 1 + 2^-7 (odd mantissa) and 1 + 2^-6 (even).
    one, up1, up2 = (int(b) for b in bf16_bits([1.0, 1.0 + 2 ** -7, 1.0 + 2 ** -6]))
    w = oracle.INTERMEDIATE_REL_WINDOW
    assert oracle.round_intermediate(1.0 + 2 ** -8, w) == (one, up1)
    assert oracle.round_intermediate(1.0 + 3 * 2 ** -8, w) == (up2, up1)
    # just inside / just outside the window, on both sides of a midpoint
    assert oracle.round_intermediate(1.0 + 2 ** -8 - 2 ** -18, w) == (one, up1)
    assert oracle.round_intermediate(1.0 + 2 ** -8 + 2 ** -18, w) == (up1, one)
    assert oracle.round_intermediate(1.0 + 2 ** -8 - 2 ** -15, w) == (one, one)
    assert oracle.round_intermediate(1.0 + 2 ** -8 + 2 ** -15, w) == (up1, up1)
    # negative values mirror
    mone, mup1 = (int(b) for b in bf16_bits([-1.0, -1.0 - 2 ** -7]))
    assert oracle.round_intermediate(-1.0 - 2 ** -8, w) == (mone, mup1)


# ------------------------------------------------------------------------------------------
# outputs without an intermediate: no window, check() is the formula
# ------------------------------------------------------------------------------------------

def _dense(M, N, K, seed):
    w = synth.fp4_bytes(N, K, seed=seed).numpy()
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=seed + 1).numpy()
    x = u16(synth.activations(M, K, seed=seed + 2))
    return x, w, sf


def test_plain_outputs_have_no_window():
    x, w, sf = _dense(4, 256, 4096, seed=61)
    nom, lo, hi = oracle.nvfp4_gemv(x, w, sf, 0.01)
    assert np.array_equal(lo, nom) and np.array_equal(hi, nom)
    wb = u16(synth.bf16_weight(128, 1024, seed=62))
    xb = u16(synth.activations(3, 1024, seed=63))
    nom, lo, hi = oracle.bf16_gemv(xb, wb)
    assert np.array_equal(lo, nom) and np.array_equal(hi, nom)


def test_routed_gate_up_has_no_window():
    from test_oracle_moe import tiny_moe
    d = tiny_moe(M=4, E=4, H=512, I=128, SI=128, topk=2, seed=7)
    (act, alo, ahi), _, bad = oracle.moe_gate_up(d["x"], d["ids"], d["w1"], d["w1_sf"], d["alpha"], d["wsh"],
                                                 d["ssh"], 0.01)
    assert bad == 0
    assert np.array_equal(alo, act) and np.array_equal(ahi, act)


def test_check_equals_formula_without_window():
    # Random perturbations of a plain output: check() flags exactly the
    # elements the written-out formula flags.
    x, w, sf = _dense(4, 512, 2048, seed=64)
    ref = oracle.nvfp4_gemv(x, w, sf, 0.01)
    nom = oracle.bf16_to_f64(ref[0])
    rng = np.random.default_rng(65)
    for scale in (2.0 ** -9, 2.0 ** -7, 2.0 ** -6, 2.0 ** -4):
        pert = nom * (1.0 + scale * rng.standard_normal(nom.shape)) + scale * rng.standard_normal(nom.shape)
        gb = bf16_bits(pert.astype(np.float32))
        ok, _, nbad, _ = oracle.check(gb, ref)
        want = int(formula_bad(gb, ref[0]).sum())
        assert nbad == want and ok == (want == 0), scale
    # one bf16 ulp off in either direction always passes
    for step in (1, -1):
        gb = (ref[0].astype(np.int32) + step * np.where(ref[0] & 0x7FFF, 1, 0)).astype(np.uint16)
        assert oracle.check(gb, ref)[0]


# ------------------------------------------------------------------------------------------
# intermediates: the window opens only next to a midpoint
# ------------------------------------------------------------------------------------------

def _independent_gate_up_values(x, w, sf, gs, K):
    """f32(f32(acc) * gs) of every row, from an independent decode and a
    float64 torch matmul."""
    N = w.shape[0]
    wd = independent_decode(w, oracle.scales_logical(sf, N, K))
    xd = oracle.bf16_to_f64(x)
    acc = torch.matmul(torch.from_numpy(xd), torch.from_numpy(wd).T).numpy()
    return (acc.astype(np.float32) * np.float32(gs)).astype(np.float32).astype(np.float64)


def test_silu_mul_window_empty_unless_intermediate_near_midpoint():
    M, N, K, gs = 4, 1024, 4096, 0.01
    x, w, sf = _dense(M, N, K, seed=66)
    nom, lo, hi = oracle.nvfp4_gemv(x, w, sf, gs, silu_mul=True)
    v = _independent_gate_up_values(x, w, sf, gs, K)
    G, U = v[:, : N // 2], v[:, N // 2:]
    near = (bf16_midpoint_distance(G) <= oracle.INTERMEDIATE_REL_WINDOW * np.abs(G)) | \
           (bf16_midpoint_distance(U) <= oracle.INTERMEDIATE_REL_WINDOW * np.abs(U))
    open_ = (lo != nom) | (hi != nom)
    assert not (open_ & ~near).any(), "a window opened with no intermediate near a midpoint"
    assert near.sum() >= 5 and open_.sum() >= 1, (int(near.sum()), int(open_.sum()))
    # where the window is open, it holds exactly the outputs of the four
    # (G, U) roundings, recomputed here
    for m, i in zip(*np.nonzero(open_)):
        cands = []
        for g in {oracle.round_intermediate(G[m, i], 2 ** -16 * abs(G[m, i]))[k] for k in (0, 1)}:
            for u in {oracle.round_intermediate(U[m, i], 2 ** -16 * abs(U[m, i]))[k] for k in (0, 1)}:
                gv, uv = oracle.bf16_value(g), oracle.bf16_value(u)
                cands.append(oracle.bf16_value(oracle.bf16_rne(gv / (1.0 + math.exp(-gv)) * uv)))
        assert oracle.bf16_value(int(lo[m, i])) == min(cands) and oracle.bf16_value(int(hi[m, i])) == max(cands)


def test_down_combine_window_empty_unless_intermediate_near_midpoint():
    from test_oracle_moe import moe_down_inputs
    d = moe_down_inputs(M=6, E=8, H=256, I=512, SI=512, topk=4, seed=300)
    M, H, I, SI, topk = d["M"], d["H"], d["I"], d["SI"], d["topk"]
    (out, lo, hi), bad = oracle.moe_down_combine(d["act"], d["ids"], d["tw"], d["w2"], d["w2_sf"], d["alpha2"],
                                                 d["sact"], d["wsd"], d["ssd"], 0.01)
    assert bad == 0
    sfe = oracle.scale_bytes(H, I)
    actd, sactd = oracle.bf16_to_f64(d["act"]), oracle.bf16_to_f64(d["sact"])
    wsd = independent_decode(d["wsd"], oracle.scales_logical(d["ssd"], H, SI))
    near = np.zeros((M, H), bool)
    for t in range(M):
        s, sabs = np.zeros(H), np.zeros(H)
        for j in range(topk):
            e = int(d["ids"][t, j])
            wd = independent_decode(d["w2"][e], oracle.scales_logical(d["w2_sf"][e * sfe:(e + 1) * sfe], H, I))
            y = ((wd @ actd[t * topk + j]).astype(np.float32) * np.float32(d["alpha2"][e])).astype(np.float64)
            near[t] |= bf16_midpoint_distance(y) <= 2 ** -16 * np.abs(y)
            yb = oracle.bf16_to_f64(bf16_bits(y.astype(np.float32)))
            s += np.float64(d["tw"][t, j]) * yb
            sabs += np.abs(np.float64(d["tw"][t, j]) * yb)
        near[t] |= bf16_midpoint_distance(s) <= (topk + 1) * 2 ** -24 * sabs
        ysh = ((wsd @ sactd[t]).astype(np.float32) * np.float32(0.01)).astype(np.float64)
        near[t] |= bf16_midpoint_distance(ysh) <= 2 ** -16 * np.abs(ysh)
    open_ = (lo != out) | (hi != out)
    assert not (open_ & ~near).any(), "a window opened with no intermediate near a midpoint"
    assert near.sum() >= 1


# ------------------------------------------------------------------------------------------
# planted mistakes at large K
# ------------------------------------------------------------------------------------------

def _flagged(got, ref):
    ok, _, nbad, _ = oracle.check(got, ref)
    return nbad / got.size


@pytest.mark.parametrize("K", [14336, 28672])
def test_planted_mistakes_fail_at_large_k(K):
    M, N, gs = 4, 128, 0.01
    x, w, sf = _dense(M, N, K, seed=K)
    ref = oracle.nvfp4_gemv(x, w, sf, gs)
    assert oracle.check(ref[0], ref)[0]
    # one 16-wide K block dropped from every row (its codes zeroed)
    w_drop = w.copy()
    w_drop[:, 8 * 37:8 * 38] = 0
    got = oracle.nvfp4_gemv(x, w_drop, sf, gs)[0]
    frac = _flagged(got, ref)
    assert frac == formula_bad(got, ref[0]).mean()  # no window: the rule is the formula
    assert frac >= 0.4, frac
    # every scale one E4M3 step up (the next code; the draws stay below 448)
    sf_up = (sf.astype(np.int32) + np.where(sf > 0, 1, 0)).astype(np.uint8)
    assert _flagged(oracle.nvfp4_gemv(x, w, sf_up, gs)[0], ref) >= 0.9
    # gate and up rows swapped (silu_mul on [gate | up] halves)
    ref_s = oracle.nvfp4_gemv(x, w, sf, gs, silu_mul=True)
    swapped = np.concatenate([w[N // 2:], w[: N // 2]])
    sf_sw = np.zeros_like(sf)
    for r in range(N):
        src = (r + N // 2) % N
        for kb in range(K // 16):
            sf_sw[oracle.swz(r, kb, K)] = sf[oracle.swz(src, kb, K)]
    assert _flagged(oracle.nvfp4_gemv(x, swapped, sf_sw, gs, silu_mul=True)[0], ref_s) >= 0.6


# ------------------------------------------------------------------------------------------
# the window's width against fp32 accumulation
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("K", [4096, 8192, 28672])
def test_window_covers_fp32_blocked_accumulation(K):
    # Emulate an fp32 accumulator that adds one 16-product block at a time
    # (each block sum rounded to fp32, then one fp32 add), sequentially over
    # all of K, the longest chain an implementation can have.  For every
    # value not small against the rms (|v| >= rms / 16) the relative error
    # stays below the intermediate window; smaller values move the output by
    # less than the tolerance's rms term when they round the other way.
    R = 384
    rng = np.random.default_rng(K)
    x = torch.from_numpy(rng.standard_normal((R, K)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    codes = rng.integers(0, 16, (R, K))
    table = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, 0, -.5, -1, -1.5, -2, -3, -4, -6])
    sc = torch.exp2(torch.from_numpy(rng.uniform(-3, 3, (R, K // 16)))).to(torch.float8_e4m3fn).double().numpy()
    p = x * table[codes] * np.repeat(sc, 16, axis=1)
    exact = p.sum(axis=1)
    blocks = p.reshape(R, -1, 16).sum(axis=2)
    acc = np.zeros(R, np.float32)
    for b in range(blocks.shape[1]):
        acc = (acc.astype(np.float64) + blocks[:, b].astype(np.float32).astype(np.float64)).astype(np.float32)
    rms = math.sqrt(float(np.mean(exact * exact)))
    big = np.abs(exact) >= rms / 16
    rel = np.abs(acc.astype(np.float64) - exact)[big] / np.abs(exact[big])
    assert rel.max() < oracle.INTERMEDIATE_REL_WINDOW, math.log2(rel.max())
