"""Pins for the oracle's MoE pair (CPU only): brute force at tiny sizes,
reductions to the dense ops, and an exact-integer routing probe."""
import math

import numpy as np
import torch

import oracle
from moe_nvfp4_gemv_gb300 import synth

from test_oracle_gemv import E2M1_TABLE, bf16_bits, independent_decode, place_scales


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def tiny_moe(M=3, E=4, H=64, I=64, SI=128, topk=2, seed=0):
    ids, tw = synth.routing(M, E, topk, seed=seed)
    x = u16(synth.activations(M, H, seed=seed + 1))
    w1 = np.stack([synth.fp4_bytes(2 * I, H, seed=seed + 10 + e).numpy() for e in range(E)])
    w1_sf = np.concatenate([synth.e4m3_bytes(oracle.scale_bytes(2 * I, H), seed=seed + 30 + e).numpy()
                            for e in range(E)])
    alpha = synth.expert_alphas(E).numpy()
    wsh = synth.fp4_bytes(2 * SI, H, seed=seed + 50).numpy()
    ssh = synth.e4m3_bytes(oracle.scale_bytes(2 * SI, H), seed=seed + 51).numpy()
    return dict(M=M, E=E, H=H, I=I, SI=SI, topk=topk, ids=ids.numpy(), tw=tw.numpy(), x=x, w1=w1,
                w1_sf=w1_sf, alpha=alpha, wsh=wsh, ssh=ssh)


def test_gate_up_brute_force():
    d = tiny_moe()
    M, E, H, I, SI, topk = (d[k] for k in ("M", "E", "H", "I", "SI", "topk"))
    xd = oracle.bf16_to_f64(d["x"])
    sfe = oracle.scale_bytes(2 * I, H)
    (act, _, _), (sact, _, _), bad = oracle.moe_gate_up(d["x"], d["ids"], d["w1"], d["w1_sf"], d["alpha"],
                                                        d["wsh"], d["ssh"], 0.01)
    assert bad == 0
    for p in range(M * topk):
        t, e = p // topk, int(d["ids"].reshape(-1)[p])
        wd = independent_decode(d["w1"][e], oracle.scales_logical(d["w1_sf"][e * sfe:(e + 1) * sfe], 2 * I, H))
        # "[up; gate] in 64-row groups": stored rows 128g..128g+63 are up rows
        # 64g..64g+63, stored rows 128g+64..128g+127 the gate rows.
        up = np.concatenate([wd[128 * g:128 * g + 64] for g in range(I // 64)])
        gate = np.concatenate([wd[128 * g + 64:128 * g + 128] for g in range(I // 64)])
        a = np.float32(d["alpha"][e])
        g = (np.float32(gate @ xd[t]) * a).astype(np.float64)
        u = (np.float32(up @ xd[t]) * a).astype(np.float64)
        want = [oracle.bf16_rne(gi / (1.0 + math.exp(-gi)) * ui) for gi, ui in zip(g, u)]
        assert act[p].tolist() == want, p
    # shared expert: the dense silu_mul GEMV on the ModelOpt [gate; up] weight
    dense, _, _ = oracle.nvfp4_gemv(d["x"], d["wsh"], d["ssh"], 0.01, silu_mul=True)
    assert np.array_equal(sact, dense)


def test_gate_up_row_map_reading():
    assert [oracle.w1_row(i, True) for i in (0, 63, 64, 127)] == [0, 63, 128, 191]
    assert [oracle.w1_row(i, False) for i in (0, 63, 64, 127)] == [64, 127, 192, 255]


def moe_down_inputs(M=3, E=4, H=128, I=64, SI=64, topk=2, seed=100):
    ids, tw = synth.routing(M, E, topk, seed=seed)
    act = u16(synth.activations(M * topk, I, seed=seed + 1))
    sact = u16(synth.activations(M, SI, seed=seed + 2))
    w2 = np.stack([synth.fp4_bytes(H, I, seed=seed + 10 + e).numpy() for e in range(E)])
    w2_sf = np.concatenate([synth.e4m3_bytes(oracle.scale_bytes(H, I), seed=seed + 30 + e).numpy()
                            for e in range(E)])
    alpha2 = synth.expert_alphas(E).numpy()
    wsd = synth.fp4_bytes(H, SI, seed=seed + 50).numpy()
    ssd = synth.e4m3_bytes(oracle.scale_bytes(H, SI), seed=seed + 51).numpy()
    return dict(ids=ids.numpy(), tw=tw.numpy(), act=act, sact=sact, w2=w2, w2_sf=w2_sf, alpha2=alpha2,
                wsd=wsd, ssd=ssd, M=M, E=E, H=H, I=I, SI=SI, topk=topk)


def test_down_combine_brute_force():
    d = moe_down_inputs()
    M, H, I, topk = d["M"], d["H"], d["I"], d["topk"]
    (out, lo, hi), bad = oracle.moe_down_combine(d["act"], d["ids"], d["tw"], d["w2"], d["w2_sf"], d["alpha2"],
                                                 d["sact"], d["wsd"], d["ssd"], 0.01)
    assert bad == 0
    sfe = oracle.scale_bytes(H, I)
    actd = oracle.bf16_to_f64(d["act"])
    sactd = oracle.bf16_to_f64(d["sact"])
    wsd = independent_decode(d["wsd"], oracle.scales_logical(d["ssd"], H, d["SI"]))
    for t in range(M):
        s = np.zeros(H)
        for j in range(topk):
            e = int(d["ids"][t, j])
            wd = independent_decode(d["w2"][e], oracle.scales_logical(d["w2_sf"][e * sfe:(e + 1) * sfe], H, I))
            acc = wd @ actd[t * topk + j]
            y = oracle.bf16_to_f64(bf16_bits((acc.astype(np.float32) * np.float32(d["alpha2"][e])).astype(np.float32)))
            s += np.float64(d["tw"][t, j]) * y
        sb = np.array([oracle.bf16_rne(v) for v in s], np.uint16)
        ysh = bf16_bits(((wsd @ sactd[t]).astype(np.float32) * np.float32(0.01)).astype(np.float32))
        want = [oracle.bf16_rne(a + b) for a, b in zip(oracle.bf16_to_f64(sb), oracle.bf16_to_f64(ysh))]
        assert out[t].tolist() == want, t
    lod, nomd, hid = oracle.bf16_to_f64(lo), oracle.bf16_to_f64(out), oracle.bf16_to_f64(hi)
    assert (lod <= nomd).all() and (nomd <= hid).all()


def test_down_combine_reduces_to_dense_gemv():
    # topk = 1, tw = 1, zero shared expert: out = y = the dense GEMV of act
    # against W2[e] with global scale alpha2[e].
    d = moe_down_inputs(M=4, topk=1, seed=200)
    d["tw"][:] = 1.0
    d["wsd"][:] = 0
    (out, _, _), bad = oracle.moe_down_combine(d["act"], d["ids"], d["tw"], d["w2"], d["w2_sf"], d["alpha2"],
                                               d["sact"], d["wsd"], d["ssd"], 0.01)
    sfe = oracle.scale_bytes(d["H"], d["I"])
    for t in range(d["M"]):
        e = int(d["ids"][t, 0])
        dense, _, _ = oracle.nvfp4_gemv(d["act"][t:t + 1], d["w2"][e], d["w2_sf"][e * sfe:(e + 1) * sfe],
                                        float(d["alpha2"][e]))
        assert np.array_equal(out[t], dense[0]), t


def test_down_combine_routing_probe_exact():
    # Expert e's W2 is 1.0 in K column 0 and 0 elsewhere, with the scale of
    # block 0 equal to 2^e; act rows are one-hot at column 0; tw = [1, 1/16];
    # alpha2 = 1; the shared expert is zero.  Then out[t, h] = 2^e0 + 2^(e1-4)
    # exactly, which identifies both experts and their weights.
    M, E, H, I, SI, topk = 5, 4, 128, 64, 64, 2
    w2 = np.zeros((E, H, I // 2), np.uint8)
    w2[:, :, 0] = 0x02  # low nibble (k = 0) = code 2 = 1.0
    sfe = oracle.scale_bytes(H, I)
    w2_sf = np.zeros(E * sfe, np.uint8)
    for e in range(E):
        logical = np.full((H, I // 16), 0x38, np.uint8)
        logical[:, 0] = 0x38 + 8 * e  # 2^e
        w2_sf[e * sfe:(e + 1) * sfe] = place_scales(logical, I)
    act = np.zeros((M * topk, I), np.uint16)
    act[:, 0] = bf16_bits([1.0])[0]
    ids = np.array([[0, 1], [3, 2], [2, 0], [1, 3], [3, 0]], np.int32)
    tw = np.tile(np.array([1.0, 1.0 / 16], np.float32), (M, 1))
    alpha2 = np.ones(E, np.float32)
    sact = np.zeros((M, SI), np.uint16)
    wsd = np.zeros((H, SI // 2), np.uint8)
    ssd = np.zeros(oracle.scale_bytes(H, SI), np.uint8)
    (out, lo, hi), bad = oracle.moe_down_combine(act, ids, tw, w2, w2_sf, alpha2, sact, wsd, ssd, 1.0)
    assert bad == 0
    for t in range(M):
        want = 2.0 ** ids[t, 0] + 2.0 ** (ids[t, 1] - 4)
        assert (oracle.bf16_to_f64(out[t]) == want).all(), t
        assert np.array_equal(lo[t], out[t]) and np.array_equal(hi[t], out[t])


def test_bad_ids_are_reported_not_used():
    d = moe_down_inputs()
    d["ids"][1, 0] = 99
    (out, _, _), bad = oracle.moe_down_combine(d["act"], d["ids"], d["tw"], d["w2"], d["w2_sf"], d["alpha2"],
                                               d["sact"], d["wsd"], d["ssd"], 0.01)
    assert bad == 1 and not out[1].any()
