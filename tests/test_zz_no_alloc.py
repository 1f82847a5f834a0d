"""fp4gemv_moe_down_combine_noalloc: down_combine for callers that cannot
allocate device memory (its scratch is a fixed array inside the library).

Called through the C ABI twice in a row and checked against the regular
fp4gemv_moe_down_combine (caller workspace) on the same inputs, within the
tolerance the parity tests use.  Kept in a file pytest collects last."""
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


def _inputs(M, E, H, I, SI, topk, seed):
    ids, tw = synth.routing(M, E, topk, seed=seed)
    d = dict(ids=ids, tw=tw, act=synth.activations(M * topk, I, seed=seed + 1),
             sact=synth.activations(M, SI, seed=seed + 2),
             w2=torch.stack([synth.fp4_bytes(H, I, seed=seed + 10 + e) for e in range(E)]),
             w2_sf=torch.cat([synth.e4m3_bytes(oracle.scale_bytes(H, I), seed=seed + 200 + e) for e in range(E)]),
             alpha2=synth.expert_alphas(E), wsd=synth.fp4_bytes(H, SI, seed=seed + 3),
             ssd=synth.e4m3_bytes(oracle.scale_bytes(H, SI), seed=seed + 4), gssd=torch.tensor([0.01]))
    return {k: v.to(DEV) for k, v in d.items()}


def _noalloc(lib, d, M, E, H, I, SI, topk, out):
    vp = ctypes.c_void_p
    p = lambda t: vp(t.data_ptr())  # noqa: E731
    f = lib.fp4gemv_moe_down_combine_noalloc
    f.restype = ctypes.c_int
    stream = vp(torch.cuda.current_stream().cuda_stream)
    return f(p(d["act"]), p(d["ids"]), p(d["tw"]), M, topk, p(d["w2"]), p(d["w2_sf"]), p(d["alpha2"]), E, H, I,
             p(d["sact"]), p(d["wsd"]), p(d["ssd"]), p(d["gssd"]), SI, p(out), 1, stream)


@pytest.mark.parametrize("shape", [dict(M=8, E=128, H=4096, I=1536, SI=1536, topk=8),
                                   dict(M=3, E=16, H=1024, I=512, SI=768, topk=2)])
def test_noalloc_matches_workspace_entry_point_twice(shape):
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from moe_nvfp4_gemv_gb300 import fp4gemv
    lib = fp4gemv.lib()
    M, E, H, I, SI, topk = (shape[k] for k in ("M", "E", "H", "I", "SI", "topk"))
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        d = _inputs(M, E, H, I, SI, topk, seed)
        ref = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
        fp4gemv.moe_down_combine(d["act"], d["ids"], d["tw"], d["w2"], d["w2_sf"], d["alpha2"], d["sact"], d["wsd"],
                                 d["ssd"], d["gssd"], ref)
        out = torch.full((M, H), 7.0, dtype=torch.bfloat16, device=DEV)
        assert _noalloc(lib, d, M, E, H, I, SI, topk, out) == 0
        torch.cuda.synchronize()
        r = _u16(ref)
        ok, excess, nbad, _ = oracle.check(_u16(out), (r, r, r))
        assert ok, f"call {call}: {nbad} elements outside tolerance (excess {excess})"
    assert fp4gemv.get_device_error() == 0


def test_noalloc_rejects_oversized_shapes():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from moe_nvfp4_gemv_gb300 import fp4gemv
    lib = fp4gemv.lib()
    limit = 8 << 20
    M, topk, H = 256, 4, 8192  # y alone is 2 * 1024 * 8192 bytes = 16 MiB
    assert fp4gemv.moe_down_combine_workspace_bytes(M, topk, H) > limit
    vp = ctypes.c_void_p
    f = lib.fp4gemv_moe_down_combine_noalloc
    f.restype = ctypes.c_int
    a = vp(1 << 20)
    assert f(a, a, a, M, topk, a, a, a, 8, H, 1536, a, a, a, a, 1536, a, 1, None) == 2
