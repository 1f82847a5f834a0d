"""fp4gemv_moe_down_combine_noalloc: down_combine for callers that cannot
allocate device memory (its scratch is a fixed array inside the library).

Called through the C ABI twice in a row, each result compared bit for bit
with the regular fp4gemv_moe_down_combine (caller workspace, the same
deterministic kernel) on the same inputs and checked against the oracle.
Also: several gate_up -> down_combine_noalloc layers chained on one stream
with programmatic dependent launch (each layer's output feeds the next), and
back-to-back down_combine calls sharing one workspace, every output checked.
Kept in a file pytest collects last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from moe_nvfp4_gemv_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _fp4():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from moe_nvfp4_gemv_gb300 import fp4gemv
    return fp4gemv


def _down_inputs(M, E, H, I, SI, topk, seed):
    ids, tw = synth.routing(M, E, topk, seed=seed)
    return dict(ids=ids, tw=tw, act=synth.activations(M * topk, I, seed=seed + 1),
                sact=synth.activations(M, SI, seed=seed + 2),
                w2=torch.stack([synth.fp4_bytes(H, I, seed=seed + 10 + e) for e in range(E)]),
                w2_sf=torch.cat([synth.e4m3_bytes(oracle.scale_bytes(H, I), seed=seed + 1000 + e) for e in range(E)]),
                alpha2=synth.expert_alphas(E), wsd=synth.fp4_bytes(H, SI, seed=seed + 3),
                ssd=synth.e4m3_bytes(oracle.scale_bytes(H, SI), seed=seed + 4), gssd=torch.tensor([0.01]))


def _noalloc(lib, d, M, E, H, I, SI, topk, out, pdl=1):
    vp = ctypes.c_void_p
    p = lambda t: vp(t.data_ptr())  # noqa: E731
    f = lib.fp4gemv_moe_down_combine_noalloc
    f.restype = ctypes.c_int
    stream = vp(torch.cuda.current_stream().cuda_stream)
    return f(p(d["act"]), p(d["ids"]), p(d["tw"]), M, topk, p(d["w2"]), p(d["w2_sf"]), p(d["alpha2"]), E, H, I,
             p(d["sact"]), p(d["wsd"]), p(d["ssd"]), p(d["gssd"]), SI, p(out), pdl, stream)


def _oracle_down(d, tokens):
    h = {k: v.numpy() if v.dtype != torch.bfloat16 else _u16(v) for k, v in d.items()}
    (ref, bad) = oracle.moe_down_combine(h["act"], h["ids"], h["tw"], h["w2"], h["w2_sf"], h["alpha2"], h["sact"],
                                         h["wsd"], h["ssd"], float(h["gssd"][0]), tokens=tokens)
    assert bad == 0
    return ref


@pytest.mark.parametrize("shape", [dict(M=8, E=128, H=4096, I=1536, SI=1536, topk=8),
                                   dict(M=3, E=16, H=1024, I=512, SI=768, topk=2)])
def test_noalloc_matches_workspace_entry_point_twice(shape):
    fp4gemv = _fp4()
    lib = fp4gemv.lib()
    M, E, H, I, SI, topk = (shape[k] for k in ("M", "E", "H", "I", "SI", "topk"))
    tokens = sorted({0, M - 1})
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        host = _down_inputs(M, E, H, I, SI, topk, seed)
        d = {k: v.to(DEV) for k, v in host.items()}
        ref = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
        fp4gemv.moe_down_combine(d["act"], d["ids"], d["tw"], d["w2"], d["w2_sf"], d["alpha2"], d["sact"], d["wsd"],
                                 d["ssd"], d["gssd"], ref)
        out = torch.full((M, H), 7.0, dtype=torch.bfloat16, device=DEV)
        assert _noalloc(lib, d, M, E, H, I, SI, topk, out) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}: the two entry points differ"
        o = _oracle_down(host, tokens)
        ok, excess, nbad, _ = oracle.check(_u16(out)[tokens], tuple(r[tokens] for r in o))
        assert ok, f"call {call}: {nbad} elements outside tolerance (excess {excess})"
    assert fp4gemv.get_device_error() == 0


def test_noalloc_chained_layers_under_pdl():
    # gate_up -> down_combine_noalloc, three layers, one stream, PDL on, the
    # output of each layer the input of the next; every launch checked.
    fp4gemv = _fp4()
    lib = fp4gemv.lib()
    M, E, H, I, SI, topk = 4, 16, 1024, 512, 512, 4
    layers = []
    for l in range(3):
        s = 100 * (l + 1)
        ids, tw = synth.routing(M, E, topk, seed=s)
        layers.append(dict(
            ids=ids, tw=tw,
            w1=torch.stack([synth.fp4_bytes(2 * I, H, seed=s + 1 + e) for e in range(E)]),
            w1_sf=torch.cat([synth.e4m3_bytes(oracle.scale_bytes(2 * I, H), seed=s + 40 + e) for e in range(E)]),
            alpha=synth.expert_alphas(E), wsh=synth.fp4_bytes(2 * SI, H, seed=s + 80),
            ssh=synth.e4m3_bytes(oracle.scale_bytes(2 * SI, H), seed=s + 81), gssh=torch.tensor([0.01]),
            w2=torch.stack([synth.fp4_bytes(H, I, seed=s + 90 + e) for e in range(E)]),
            w2_sf=torch.cat([synth.e4m3_bytes(oracle.scale_bytes(H, I), seed=s + 130 + e) for e in range(E)]),
            alpha2=synth.expert_alphas(E), wsd=synth.fp4_bytes(H, SI, seed=s + 170),
            ssd=synth.e4m3_bytes(oracle.scale_bytes(H, SI), seed=s + 171), gssd=torch.tensor([0.01])))
    dl = [{k: v.to(DEV) for k, v in L.items()} for L in layers]
    x0 = synth.activations(M, H, seed=7).to(DEV)
    xs, acts, sacts, outs = [x0], [], [], []
    for d in dl:  # all launches queued back to back, no host synchronisation
        act = torch.empty(M * topk, I, dtype=torch.bfloat16, device=DEV)
        sact = torch.empty(M, SI, dtype=torch.bfloat16, device=DEV)
        fp4gemv.moe_gate_up(xs[-1], d["ids"], d["w1"], d["w1_sf"], d["alpha"], act, d["wsh"], d["ssh"], d["gssh"],
                            sact, pdl=True)
        out = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
        dd = dict(act=act, ids=d["ids"], tw=d["tw"], w2=d["w2"], w2_sf=d["w2_sf"], alpha2=d["alpha2"], sact=sact,
                  wsd=d["wsd"], ssd=d["ssd"], gssd=d["gssd"])
        assert _noalloc(lib, dd, M, E, H, I, SI, topk, out, pdl=1) == 0
        acts.append(act)
        sacts.append(sact)
        outs.append(out)
        xs.append(out)
    torch.cuda.synchronize()
    for l, L in enumerate(layers):
        h = {k: v.numpy() for k, v in L.items()}
        (a_ref, s_ref, bad) = oracle.moe_gate_up(_u16(xs[l]), h["ids"], h["w1"], h["w1_sf"], h["alpha"], h["wsh"],
                                                 h["ssh"], 0.01)
        assert bad == 0
        assert oracle.check(_u16(acts[l]), a_ref)[0], f"layer {l} act"
        assert oracle.check(_u16(sacts[l]), s_ref)[0], f"layer {l} sact"
        d = dict(L, act=acts[l].cpu(), sact=sacts[l].cpu())
        o = _oracle_down(d, list(range(M)))
        ok, excess, nbad, _ = oracle.check(_u16(outs[l]), o)
        assert ok, f"layer {l} out: {nbad} outside tolerance (excess {excess})"
    assert fp4gemv.get_device_error() == 0


# (8 tokens over 32 experts: one CTA per item, one wave; 16 tokens over 128
# experts: the persistent grid, whose work counter each call restarts)
@pytest.mark.parametrize("M,E", [(8, 32), (16, 128)])
def test_back_to_back_down_combine_share_a_workspace(M, E):
    # Consecutive down_combine launches with PDL and one workspace: each
    # call's counters (abort tags, the persistent grid's work counter) must be
    # out of use before the next call claims them.  Every output is compared
    # with its own isolated run.
    fp4gemv = _fp4()
    H, I, SI, topk = 2048, 512, 512, 8
    ins = [{k: v.to(DEV) for k, v in _down_inputs(M, E, H, I, SI, topk, seed).items()} for seed in (21, 22, 23, 24)]
    ws = torch.empty(fp4gemv.moe_down_combine_workspace_bytes(M, topk, H), dtype=torch.uint8, device=DEV)
    iso = []
    for d in ins:
        o = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
        fp4gemv.moe_down_combine(d["act"], d["ids"], d["tw"], d["w2"], d["w2_sf"], d["alpha2"], d["sact"], d["wsd"],
                                 d["ssd"], d["gssd"], o, pdl=False, workspace=ws)
        torch.cuda.synchronize()
        iso.append(o)
    for rep in range(3):
        outs = [torch.full((M, H), 3.0, dtype=torch.bfloat16, device=DEV) for _ in ins]
        for d, o in zip(ins, outs):
            fp4gemv.moe_down_combine(d["act"], d["ids"], d["tw"], d["w2"], d["w2_sf"], d["alpha2"], d["sact"],
                                     d["wsd"], d["ssd"], d["gssd"], o, pdl=True, workspace=ws)
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(outs, iso)):
            assert torch.equal(a, b), f"repeat {rep}, call {i}"
    assert fp4gemv.get_device_error() == 0


def test_noalloc_rejects_oversized_shapes():
    # Null pointers throughout: the size check comes first; if it regressed,
    # the null-pointer check would return FP4GEMV_ERR_INVALID_ARG, never a
    # launch.
    fp4gemv = _fp4()
    lib = fp4gemv.lib()
    limit = 8 << 20
    M, topk, H = 256, 4, 8192  # y alone is 2 * 1024 * 8192 bytes = 16 MiB
    assert fp4gemv.moe_down_combine_workspace_bytes(M, topk, H) > limit
    vp = ctypes.c_void_p
    f = lib.fp4gemv_moe_down_combine_noalloc
    f.restype = ctypes.c_int
    z = vp(0)
    assert f(z, z, z, M, topk, z, z, z, 8, H, 1536, z, z, z, z, 1536, z, 1, None) == 2
