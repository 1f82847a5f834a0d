"""The timeout path on the GPU, made without a fault: the dense GEMV's
producers are told (a host-side test hook) to issue nothing for one ring
stage -- no copy and no arrival, so nothing is in flight when a wait gives
up -- and the wait limit is lowered to a few milliseconds.  The call must
come back, the device error word must read FP4GEMV_ERR_TIMEOUT, the outputs
must be left unwritten, and the next normal call must be correct.  Unsplit
(one CTA per cluster) launches on both kernels that serve 1 .. 16 tokens,
and down_combine on the slab kernel, whose CTAs that gave up tag their row
tiles so that the combine kernel after them leaves those outputs unwritten
(on both of its grids: one CTA per item, and the persistent one)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, dense_inputs, require_gpu, u16

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT = 5


@pytest.fixture()
def fp4():
    require_gpu()
    from moe_nvfp4_gemv_gb300 import fp4gemv
    yield fp4gemv
    fp4gemv.debug_skip_stage(-1)
    fp4gemv.set_wait_limit_ns(0)


def _plan_split(fp4, M, N, K):
    """The split the library picks (host-only plan functions), to make sure
    the launch under test is unsplit."""
    import ctypes
    from test_plan import GB300_CAP, Plan, SlabPlan
    lib = fp4.lib()
    regs = (ctypes.c_int * 2)(107, 125)
    sp = SlabPlan()
    f = lib.fp4gemv_plan_slab
    f.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(SlabPlan)]
    if f(M, N, K, 0, 152, regs, ctypes.byref(sp)) == 0:
        return "slab", sp.split
    rp = Plan()
    g = lib.fp4gemv_plan_rf
    g.argtypes = [ctypes.c_int] * 4 + [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(Plan)]
    assert g(N, K, 0, 152, (ctypes.c_int * 9)(*GB300_CAP), ctypes.byref(rp)) == 0
    return "rf", rp.split


@pytest.mark.parametrize("M,N,K,kernel,skip", [(1, 128, 256, "rf", 0), (5, 256, 256, "rf", 0), (12, 384, 256, "rf", 0),
                                               (1, 38912, 1024, "rf", 2), (1, 46848, 256, "slab", 0)])
def test_timeout_path_then_recovery(fp4, M, N, K, kernel, skip):
    assert _plan_split(fp4, M, N, K) == (kernel, 1)
    x, w, sf = dense_inputs(M, N, K, seed=N + M)
    xd, wd, sd = x.to(DEV), w.to(DEV), sf.to(DEV)
    gs = torch.tensor([0.01], device=DEV)
    assert fp4.get_device_error() == 0
    fp4.set_wait_limit_ns(5_000_000)  # 5 ms
    fp4.debug_skip_stage(skip)
    out = torch.full((M, N), 3.0, dtype=torch.bfloat16, device=DEV)
    fp4.nvfp4_gemv(xd, wd, sd, gs, out=out)
    assert fp4.get_device_error() == TIMEOUT  # (synchronizes; clears the word)
    assert (out == 3.0).all(), "outputs of a call that timed out must be left unwritten"
    fp4.debug_skip_stage(-1)
    fp4.set_wait_limit_ns(0)
    got = fp4.nvfp4_gemv(xd, wd, sd, gs)
    torch.cuda.synchronize()
    assert fp4.get_device_error() == 0
    rows = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N)])) if N > 512 else None
    ref = oracle.nvfp4_gemv(u16(x), w.numpy(), sf.numpy(), 0.01, rows=rows)
    g = u16(got) if rows is None else u16(got)[:, rows]
    assert_close(g, ref, f"after the timeout M={M} N={N} K={K}")


def test_skip_hook_rejects_bad_stage(fp4):
    with pytest.raises(Exception):
        fp4.debug_skip_stage(-2)


# (I = 512: two 256-K stages per row tile; SI = 256: the shared expert's
# CTAs have one, so skipping stage 1 stops only the routed CTAs.  The third
# case streams two tiles per CTA and stops in the second: the CTA has
# written the first tile's y rows, and both of its tiles are tagged.  The
# last runs on the persistent grid (items of two tiles) and stops in a CTA's
# second item, after its first item's y rows are written.)
@pytest.mark.parametrize("M,E,H,topk,T,skip", [(1, 16, 512, 2, 1, 1), (8, 16, 512, 2, 1, 0), (8, 128, 1024, 8, 2, 3),
                                               (8, 128, 4096, 8, 2, 5)])
def test_down_combine_timeout_then_recovery(fp4, M, E, H, topk, T, skip):
    from test_gpu_moe import _down_slab_tiles, make_moe, ref_down, run_down
    I, SI = 512, 256
    assert _down_slab_tiles(fp4, M, topk, E, H, I, SI) == T
    d = make_moe(M, E=E, H=H, I=I, SI=SI, topk=topk, seed=77 + M)
    assert fp4.get_device_error() == 0
    fp4.set_wait_limit_ns(5_000_000)  # 5 ms
    fp4.debug_skip_stage(skip)
    out = run_down(fp4, d)  # (filled with 7.0 before the call)
    assert fp4.get_device_error() == TIMEOUT
    assert (out == 7.0).all(), "outputs of a call that timed out must be left unwritten"
    fp4.debug_skip_stage(-1)
    fp4.set_wait_limit_ns(0)
    out = run_down(fp4, d)
    torch.cuda.synchronize()
    assert fp4.get_device_error() == 0
    ref, bad = ref_down(d)
    assert bad == 0
    assert_close(u16(out), ref, f"down_combine after the timeout M={M}")
