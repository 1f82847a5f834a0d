"""The dense GEMV's launch plan for M <= 16 (fp4gemv_plan_rf, host only): the
tile heights and K splits the library launches for the decode layers on
GB300's co-resident CTA counts, and the invariants the kernel relies on for
any shape (grid size, room for every scale group a tile's boxes touch)."""
import ctypes

import numpy as np
import pytest

# CTAs that fit on a GB300 at once in whole clusters of 1 .. 8 CTAs of the
# register-fed kernel (two per SM, 152 SMs; clusters stay inside one GPC),
# as the occupancy API reports them.
GB300_CAP = [0, 304, 304, 291, 296, 290, 276, 266, 288]
SMS = 152


class Plan(ctypes.Structure):
    _fields_ = [("tile_rows", ctypes.c_int), ("split", ctypes.c_int), ("ctas", ctypes.c_int),
                ("scale_groups", ctypes.c_int)]


@pytest.fixture(scope="module")
def plan_fn():
    from moe_nvfp4_gemv_gb300 import fp4gemv
    f = fp4gemv.lib().fp4gemv_plan_rf
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                  ctypes.POINTER(Plan)]

    def plan(N, K, silu, cap=GB300_CAP, sms=SMS):
        c = (ctypes.c_int * 9)(*cap)
        out = Plan()
        st = f(N, K, silu, sms, c, ctypes.byref(out))
        return st, out
    return plan


@pytest.mark.parametrize("N,K,silu,rows,split,ctas", [
    (28672, 4096, 1, 96, 1, 299),    # Llama-3-8B gate_up: 224 tiles of 128 rows would leave SMs uneven
    (6144, 4096, 0, 128, 4, 192),    # qkv
    (4096, 4096, 0, 128, 8, 256),    # o_proj
    (4096, 14336, 0, 128, 8, 256),   # down
    (10240, 8192, 0, 96, 2, 214),    # Llama-3-70B qkv: 160 CTAs of 128 rows leave half the slots empty
    (57344, 8192, 1, 128, 2, 896),   # Llama-3-70B gate_up: several waves at any height, the default stays
])
def test_decode_layer_plans(plan_fn, N, K, silu, rows, split, ctas):
    st, p = plan_fn(N, K, silu)
    assert st == 0
    assert (p.tile_rows, p.split, p.ctas) == (rows, split, ctas)


def test_rejects_bad_arguments(plan_fn):
    assert plan_fn(4096, 4096, 0, sms=0)[0] == 1
    assert plan_fn(4096, 4096, 2)[0] == 1
    assert plan_fn(4104, 4096, 0)[0] == 2   # N % 16
    assert plan_fn(4112, 4096, 1)[0] == 2   # silu_mul: N % 32
    assert plan_fn(4096, 4100, 0)[0] == 2   # K % 64
    assert plan_fn(4096, 128, 0)[0] == 2    # K < 256


def _groups_touched(N, silu, rows, tile):
    """128-row scale groups the tile's boxes touch (weight rows < N only)."""
    groups_total = (N + 127) // 128
    h = rows // 2 if silu else rows
    starts = [tile * h] + ([N // 2 + tile * h] if silu else [])
    n = 0
    for r0 in starts:
        g0, g1 = r0 // 128, (r0 + h - 1) // 128
        n += (g0 < groups_total) + (g1 != g0 and g1 < groups_total)
    return n


@pytest.mark.parametrize("silu", [0, 1])
def test_plan_invariants(plan_fn, silu):
    rng = np.random.default_rng(7)
    Ns = [int(v) * 32 for v in rng.integers(1, 2000, 60)] + [28672, 57344, 14336 * 2, 6144, 10240]
    Ks = [256, 320, 1024, 4096, 8192, 14336, 28672]
    for N in Ns:
        for K in Ks:
            st, p = plan_fn(N, K, silu)
            assert st == 0
            assert p.tile_rows in (96, 112, 128) and (not silu or p.tile_rows % 32 == 0)
            assert p.split in (1, 2, 4, 8)
            n_out = N // 2 if silu else N
            feats = p.tile_rows // 2 if silu else p.tile_rows
            tiles = -(-n_out // feats)
            assert p.ctas == tiles * p.split
            # every rank keeps a non-empty K range
            kslab = (-(-K // p.split) + 63) // 64 * 64
            assert (p.split - 1) * kslab < K
            # a lower tile is only chosen when its grid fits on the GPU at once
            if p.tile_rows < 128:
                assert p.ctas <= GB300_CAP[p.split]
            # room for every scale group any tile's boxes touch
            assert 1 <= p.scale_groups <= 4
            assert max(_groups_touched(N, silu, p.tile_rows, t) for t in range(tiles)) <= p.scale_groups
