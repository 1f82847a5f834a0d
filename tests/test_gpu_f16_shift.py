"""GPU parity of the slab kernel's shifted f16 route.  Each 256-K stage of
activations gets a power-of-two shift s (0 .. 14) that brings its values into
f16's normal range, and the weight scales are multiplied by 2^-s; the
products, and so the results, must be those of the unshifted arithmetic.

The activations here are grouped by stage into magnitude classes from ~1e-7
to ~1e2, each of which needs its own shift, plus one stage whose range is
wider than f16's (the bf16 route).  The weight scales reach the e4m3
subnormals, and a block of rows has only subnormal scales: with a large shift
their weights e2m1 * e4m3 * 2^-s are f16 subnormals in the MMA, so a flush to
zero anywhere would zero those rows' outputs."""
import numpy as np
import pytest
import torch

import oracle
from moe_nvfp4_gemv_gb300 import synth
from gpu_util import assert_close, require_gpu, u16

pytestmark = pytest.mark.gpu
DEV = "cuda"

# log10 magnitude of each stage class; the last mixes 1e-7 and 1e3 in one stage
CLASSES = (-6.5, -3.5, -1.0, 1.5, None)
SUB_ROWS = 16  # rows 0 .. 15: every scale an e4m3 subnormal


@pytest.fixture(scope="module")
def fp4():
    require_gpu()
    from moe_nvfp4_gemv_gb300 import fp4gemv
    return fp4gemv


def staged_activations(M, K, seed):
    """bf16 [M, K]: sign * (0.1 + |N(0, 1)|) * 10^U, U fixed per 256-K stage
    by CLASSES (cycling); the mixed class draws 1e-7 or 1e3 at random."""
    g = torch.Generator().manual_seed(seed)
    mag = 0.1 + torch.randn(M, K, generator=g).abs()
    sign = torch.where(torch.rand(M, K, generator=g) < 0.5, -1.0, 1.0)
    u = torch.empty(M, K)
    for s in range(-(-K // 256)):
        c = CLASSES[s % len(CLASSES)]
        blk = slice(256 * s, min(K, 256 * (s + 1)))
        if c is None:
            pick = torch.rand(M, blk.stop - blk.start, generator=g) < 0.5
            u[:, blk] = torch.where(pick, torch.tensor(-7.0), torch.tensor(3.0))
        else:
            u[:, blk] = c
    return (sign * mag * torch.pow(10.0, u)).to(torch.bfloat16)


def subnormal_heavy_scales(rows, K, seed):
    """Scale bytes of e4m3(2^U), U ~ Uniform[-9.5, 8.8] (zero, subnormals
    2^-9 .. 7 x 2^-9, normals up to 448), rows 0 .. SUB_ROWS - 1 all
    subnormal (bytes 1 .. 7)."""
    sf = synth.e4m3_bytes(oracle.scale_bytes(rows, K), seed=seed, lo=-9.5, hi=8.8).numpy().copy()
    rng = np.random.RandomState(seed)
    for r in range(min(rows, SUB_ROWS)):
        for kb in range(K // 16):
            sf[oracle.swz(r, kb, K)] = rng.randint(1, 8)
    return torch.from_numpy(sf)


def _dense_slab_split(fp4, M, N, K, silu):
    import ctypes
    from test_plan import SlabPlan
    f = fp4.lib().fp4gemv_plan_slab
    f.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(SlabPlan)]
    sp = SlabPlan()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    regs = (ctypes.c_int * 2)(107, 125)
    return sp.split if f(M, N, K, int(silu), sms, regs, ctypes.byref(sp)) == 0 else None


@pytest.mark.parametrize("M", [1, 2, 4])
@pytest.mark.parametrize("silu", [False, True])
def test_dense_slab_shifted_f16(fp4, M, silu):
    N, K = 28672, 1280
    assert _dense_slab_split(fp4, M, N, K, silu) is not None  # the slab kernel serves it
    x = staged_activations(M, K, seed=10 + M)
    w = synth.fp4_bytes(N, K, seed=20 + M)
    sf = subnormal_heavy_scales(N, K, seed=30 + M)
    gs = 0.5
    got = fp4.nvfp4_gemv(x.to(DEV), w.to(DEV), sf.to(DEV), torch.tensor([gs], device=DEV), silu_mul=silu)
    n_out = N // 2 if silu else N
    rng = np.random.RandomState(M)
    rows = np.unique(np.concatenate([np.arange(64), rng.choice(n_out, 128, replace=False)]))
    ref = oracle.nvfp4_gemv(u16(x), w.numpy(), sf.numpy(), gs, silu_mul=silu, rows=rows)
    assert_close(u16(got)[:, rows], ref, f"shifted f16 dense M={M} silu={silu}")
    if not silu:
        # the all-subnormal-scale rows are not flushed to zero
        assert (u16(got)[:, :SUB_ROWS] & 0x7FFF).astype(bool).any(axis=1).all()
    assert fp4.get_device_error() == 0


@pytest.mark.parametrize("M", [1, 3, 8])
def test_moe_slab_shifted_f16(fp4, M):
    from test_gpu_moe import _down_slab_tiles, _moe_slab_plan, make_moe, ref_down, ref_gate_up, run_down, run_gate_up
    E, H, I, SI, topk = 16, 1280, 1280, 512, 4
    assert _moe_slab_plan(fp4, M, topk, E, H, I, SI) is not None
    assert _down_slab_tiles(fp4, M, topk, E, H, I, SI) is not None
    d = make_moe(M, E=E, H=H, I=I, SI=SI, topk=topk, seed=40 + M)
    d["x"] = staged_activations(M, H, seed=50 + M)
    d["w1_sf"] = torch.cat([subnormal_heavy_scales(2 * I, H, seed=60 + e) for e in range(E)])
    d["act"] = staged_activations(M * topk, I, seed=70 + M)
    d["w2_sf"] = torch.cat([subnormal_heavy_scales(H, I, seed=80 + e) for e in range(E)])
    act, sact = run_gate_up(fp4, d)
    (an, al, ah), (sn, sl, sh), bad = ref_gate_up(d)
    assert bad == 0
    assert_close(u16(act), (an, al, ah), f"shifted f16 gate_up act M={M}")
    assert_close(u16(sact), (sn, sl, sh), f"shifted f16 gate_up sact M={M}")
    out = run_down(fp4, d)
    ref, bad = ref_down(d)
    assert bad == 0
    assert_close(u16(out), ref, f"shifted f16 down_combine M={M}")
    assert fp4.get_device_error() == 0
