"""The dense GEMV's launch plans (host only): fp4gemv_plan_slab for M <= 8,
fp4gemv_plan_rf for M <= 16 otherwise.  For plan_rf: the
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


# ---------------------------------------------------------------------------
# The tcgen05 kernel's plan (fp4gemv_plan_tc): NVFP4 M > 16 and BF16 weights.

class TcPlan(ctypes.Structure):
    _fields_ = [("tokens_tile", ctypes.c_int), ("ctas_per_sm", ctypes.c_int), ("tiles", ctypes.c_int),
                ("split", ctypes.c_int), ("k_slab", ctypes.c_int), ("weight_stages", ctypes.c_int),
                ("act_slots", ctypes.c_int), ("scale_slots", ctypes.c_int), ("inbox_in_ring", ctypes.c_int),
                ("smem_bytes", ctypes.c_size_t)]


@pytest.fixture(scope="module")
def tc_plan_fn():
    from moe_nvfp4_gemv_gb300 import fp4gemv
    f = fp4gemv.lib().fp4gemv_plan_tc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 6 + [ctypes.POINTER(TcPlan)]

    def plan(M, N, K, silu, bf16=0, sms=SMS):
        out = TcPlan()
        st = f(M, N, K, silu, bf16, sms, ctypes.byref(out))
        return st, out
    return plan


@pytest.mark.parametrize("name,N,K,silu,split", [
    ("8B gate_up", 28672, 4096, 1, 2),    # 224 tiles > 152 SMs: a split of two evens the load
    ("8B qkv", 6144, 4096, 0, 4),
    ("8B o_proj", 4096, 4096, 0, 8),
    ("8B down", 4096, 14336, 0, 8),
    ("70B gate_up", 57344, 8192, 1, 2),
    ("70B qkv", 10240, 8192, 0, 2),
])
def test_tc_decode_layer_splits(tc_plan_fn, name, N, K, silu, split):
    st, p = tc_plan_fn(32, N, K, silu)
    assert st == 0 and p.split == split, name


def _tc_cases():
    rng = np.random.RandomState(5)
    cases = [(M, N, K, s, b) for M in (17, 32, 33, 64, 65, 128) for (N, K) in
             ((28672, 4096), (6144, 4096), (4096, 14336), (1056, 320), (96, 2304)) for s in (0, 1) for b in (0, 1)]
    for _ in range(60):
        cases.append((int(rng.randint(17, 129)), 32 * int(rng.randint(1, 1800)), 64 * int(rng.randint(4, 400)),
                      int(rng.randint(0, 2)), int(rng.randint(0, 2))))
    return cases


@pytest.mark.parametrize("M,N,K,silu,bf16", _tc_cases())
def test_tc_plan_invariants(tc_plan_fn, M, N, K, silu, bf16):
    st, p = tc_plan_fn(M, N, K, silu, bf16)
    assert st == 0
    nt = 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128
    assert p.tokens_tile == nt
    # tensor memory: accumulator + A slots (3 up to 64 tokens, 6 above)
    assert p.ctas_per_sm == (1 if (not bf16 and nt == 128) else 2)
    n_out = N // 2 if silu else N
    assert p.tiles == -(-n_out // (64 if silu else 128))
    # the K split: ranks 1 .. 8, each with a non-empty range of whole atoms
    assert 1 <= p.split <= 8 and p.k_slab % 64 == 0
    assert (p.split - 1) * p.k_slab < K <= p.split * p.k_slab
    assert 2 <= p.weight_stages <= 8
    assert p.inbox_in_ring == (p.split == 1)
    # shared memory: within one CTA's share (two CTAs per SM leave room for
    # the kernel's static shared memory and the per-CTA reserve)
    assert p.smem_bytes <= (110 * 1024 + 1024 if p.ctas_per_sm == 2 else 227 * 1024)
    if bf16:
        assert p.act_slots == 0 and p.scale_slots == 0
    else:
        assert p.scale_slots == ((2 if (N // 2) % 64 == 0 else 3) if silu else 1)
        # activation slots: even (each warpgroup owns its slots) or 3 only
        # with three tensor-memory slots (up to 64 tokens)
        assert p.act_slots in (2, 3, 4) and (p.act_slots != 3 or nt <= 64)
        ring = p.weight_stages * (16384 + 2048 * p.scale_slots) + p.act_slots * nt * 256
        assert ring + 1024 <= p.smem_bytes


def test_tc_plan_rejects(tc_plan_fn):
    assert tc_plan_fn(16, 4096, 4096, 0)[0] == 2      # NVFP4 M <= 16: the register-fed kernel
    assert tc_plan_fn(16, 4096, 4096, 0, bf16=1)[0] == 0
    assert tc_plan_fn(129, 4096, 4096, 0)[0] == 2     # M > 128
    assert tc_plan_fn(32, 4104, 4096, 0)[0] == 2      # N % 16
    assert tc_plan_fn(32, 4096, 4096, 2)[0] == 1
    assert tc_plan_fn(32, 4096, 4096, 0, bf16=2)[0] == 1
    assert tc_plan_fn(32, 4096, 4096, 0, sms=0)[0] == 1


# --- the slab kernel's plan (M <= 8), host only ------------------------------------------

class SlabPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("row_blocks", "warps", "tile_rows", "split", "ctas", "k_slab", "stages",
                                            "slab_bytes", "ctas_per_sm")] + [("smem_bytes", ctypes.c_size_t)]


REGS = (107, 125)  # registers per thread of the two builds (only their CTA-per-SM bound matters here)


@pytest.fixture(scope="module")
def slab_fn():
    from moe_nvfp4_gemv_gb300 import fp4gemv
    f = fp4gemv.lib().fp4gemv_plan_slab
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(SlabPlan)]

    def plan(M, N, K, silu, regs=REGS, sms=SMS):
        r = (ctypes.c_int * 2)(*regs)
        out = SlabPlan()
        return f(M, N, K, silu, sms, r, ctypes.byref(out)), out
    return plan


def slab_rule(M, N, K, silu, sms=SMS):
    """The rule written out: M <= 4 and >= 1.2 tiles per SM; 128-row tiles,
    three CTAs per SM, the largest split of one wave that fills >= 2.4 CTAs
    per SM, two 256-K stages, the activation slab M x K-slab bf16 -- all
    within a third of 228 KB."""
    trows, occ = 128, 3
    h = trows // 2 if silu else trows
    tiles = -(-(N // 2 if silu else N) // h)
    if M > 4 or tiles < 1.2 * sms:
        return None
    groups = 1 + (1 if (N // 2) % h == 0 else 2) if silu else 1
    stage = -(-(trows * 128 + groups * 2048) // 1024) * 1024
    dyn = 228 * 1024 // occ - 2048
    inbox = 8 * 144 * 4
    for S in (8, 4, 2, 1):
        if tiles * S > occ * sms:
            continue
        if tiles * S < 2.4 * sms:
            return None
        kslab = -(-(-(-K // S)) // 64) * 64
        if S > 1 and (kslab < 256 or (S - 1) * kslab >= K):
            continue
        nst = -(-kslab // 256)
        slab = -(-(M * nst * 512) // 1024) * 1024
        smem = 1024 + slab + 2 * stage + inbox
        if smem > dyn:
            return None
        return dict(split=-(-K // kslab), ctas=tiles * -(-K // kslab), k_slab=kslab, stages=2, slab_bytes=slab,
                    smem_bytes=smem)
    return None


@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("N,K,silu", [(6144, 4096, 0), (4096, 4096, 0), (28672, 4096, 1), (4096, 14336, 0),
                                      (57344, 8192, 1), (8192, 28672, 0), (10240, 8192, 0), (8192, 8192, 0),
                                      (2048, 2304, 0), (1056, 1280, 1)])
def test_slab_plan_matches_rule(slab_fn, M, N, K, silu):
    st, p = slab_fn(M, N, K, silu)
    want = slab_rule(M, N, K, silu)
    if want is None:
        assert st == 2
        return
    assert st == 0
    got = dict(split=p.split, ctas=p.ctas, k_slab=p.k_slab, stages=p.stages, slab_bytes=p.slab_bytes,
               smem_bytes=p.smem_bytes)
    assert got == want
    assert (p.row_blocks, p.warps, p.tile_rows, p.ctas_per_sm) == (2, 4, 128, 3)
    # every rank has a non-empty K range and the slab holds the rank's K
    assert (p.split - 1) * p.k_slab < K and p.slab_bytes >= M * p.k_slab * 2


@pytest.mark.parametrize("M,N,K,silu,split,ctas", [
    (1, 28672, 4096, 1, 2, 448),    # Llama-3-8B gate_up
    (4, 28672, 4096, 1, 2, 448),    # gate_up at 4 tokens
    (1, 57344, 8192, 1, 1, 448),    # Llama-3-70B gate_up
])
def test_slab_plan_decode_layers(slab_fn, M, N, K, silu, split, ctas):
    st, p = slab_fn(M, N, K, silu)
    assert st == 0 and (p.split, p.ctas) == (split, ctas)


@pytest.mark.parametrize("M,N,K,silu", [(1, 4096, 4096, 0), (1, 4096, 14336, 0), (1, 6144, 4096, 0),
                                        (8, 28672, 4096, 1), (2, 57344, 8192, 1)])
def test_slab_plan_declines(slab_fn, M, N, K, silu):
    # o_proj, down, qkv: too few tiles; 8 tokens: beyond the slab kernel's
    # range; 70B gate_up at 2 tokens: the 32 KB slab does not fit beside two
    # stages at three CTAs per SM
    assert slab_fn(M, N, K, silu)[0] == 2


def test_slab_plan_rejects_bad_arguments(slab_fn):
    assert slab_fn(9, 4096, 4096, 0)[0] == 2
    assert slab_fn(0, 4096, 4096, 0)[0] == 1
    assert slab_fn(1, 4096, 4096, 2)[0] == 1
    assert slab_fn(1, 4096, 4096, 0, sms=0)[0] == 1


# --- the slab kernel's MoE gate_up plan, host only ----------------------------------------

class MoeSlabPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("split", "k_slab", "tiles_per_cta", "groups", "chunk_pairs", "columns",
                                            "tiles", "slab_bytes", "stage_bytes", "stages", "ctas_per_sm")] + \
        [("smem_bytes", ctypes.c_size_t)]


@pytest.fixture(scope="module")
def moe_slab_fn():
    from moe_nvfp4_gemv_gb300 import fp4gemv
    f = fp4gemv.lib().fp4gemv_plan_moe_slab
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 8 + [ctypes.POINTER(MoeSlabPlan)]

    def plan(M, topk, E, H, I, SI, regs=125, sms=SMS):
        out = MoeSlabPlan()
        return f(M, topk, E, H, I, SI, sms, regs, ctypes.byref(out)), out
    return plan


def moe_slab_rule(M, topk, E, H, I, SI, sms=SMS):
    """The rule written out.  Split form: chunks of <= 4 pairs; the routed
    columns that can be active (min(P, E)) and the shared expert's ceil(M / 4)
    chunks, in 128-row tiles, fit one wave at three CTAs per SM with the
    largest split whose ranks keep >= 256 of H; a CTA's slab (min(P, 4) rows of
    its H range, bf16) and two 20 KB stages fit a third of 228 KB.  Grouped
    form (M <= 64): the whole H, T = 1 tile per CTA up to 2 tokens else 2;
    chunks of 1 (M <= 2), 2 (M < 32) or 4 pairs, halved while fewer than two
    20 KB stages fit; three CTAs per SM, two from 32 tokens; as many stages
    as fit (<= 8, <= T stages of H).  For 3 <= M < 32, with n(T, c) the
    expected streaming CTAs (expected distinct experts of P uniform draws, at
    least ceil(P / c), plus ceil(M / c), times ceil(tiles / T)) and
    f = n(2, 2) / (3 sms): f < 0.7 and n(2, 4) <= 2 sms gives T = 2, pairs of
    4, two CTAs per SM; 0.9 < f <= 1.35 gives T = 1."""
    if M > 64:
        return None
    P = M * topk
    tiles = max(I // 64, -(-SI // 64))
    ctas1 = min(P, E) * (I // 64) + -(-M // 4) * -(-SI // 64)
    rows = min(P, 4)
    dyn = 228 * 1024 // 3 - 2048
    for S in (8, 4, 2, 1):
        if ctas1 * S > 3 * sms:
            continue
        kslab = -(-(-(-H // S)) // 64) * 64
        if S > 1 and (kslab < 256 or (S - 1) * kslab >= H):
            continue
        slab = -(-(rows * -(-kslab // 256) * 512) // 1024) * 1024
        smem = 1024 + slab + 2 * 20480 + 8 * 144 * 4
        if smem > dyn:
            break
        return dict(split=-(-H // kslab), k_slab=kslab, tiles_per_cta=0, groups=tiles * -(-H // kslab),
                    chunk_pairs=4, slab_bytes=slab, stages=2, ctas_per_sm=3, smem_bytes=smem)
    nst = -(-H // 256)
    occ = 2 if M >= 32 else 3
    T = 1 if M <= 2 else 2
    chunk = 4 if M >= 32 else 1 if M <= 2 else 2
    if 3 <= M < 32:
        d = E * (1.0 - (1.0 - 1.0 / E) ** P)
        n = lambda T_, c: (max(d, float(-(-P // c))) + -(-M // c)) * -(-tiles // T_)  # noqa: E731
        f = n(2, 2) / (3.0 * sms)
        if f < 0.7 and n(2, 4) <= 2.0 * sms:
            T, chunk, occ = 2, 4, 2
        elif 0.9 < f <= 1.35:
            T = 1
    while chunk >= 1:
        rows = min(P, chunk)
        slab = -(-(rows * nst * 512) // 1024) * 1024
        ns = min(8, (228 * 1024 // occ - 2048 - 1024 - slab - 8 * 144 * 4) // 20480, T * nst)
        if ns >= 2:
            return dict(split=1, k_slab=H, tiles_per_cta=T, groups=-(-tiles // T), chunk_pairs=chunk, slab_bytes=slab,
                        stages=ns, ctas_per_sm=occ, smem_bytes=1024 + slab + ns * 20480 + 8 * 144 * 4)
        chunk //= 2
    return None


@pytest.mark.parametrize("M,topk,E,H,I,SI", [(1, 8, 128, 4096, 1536, 1536), (2, 8, 128, 4096, 1536, 1536),
                                             (8, 8, 128, 4096, 1536, 1536), (32, 8, 128, 4096, 1536, 1536),
                                             (64, 8, 128, 4096, 1536, 1536), (65, 8, 128, 4096, 1536, 1536),
                                             (1, 2, 8, 512, 256, 384), (3, 2, 8, 1024, 256, 384),
                                             (2, 4, 4, 2048, 256, 256), (1, 1, 2, 256, 64, 64),
                                             (4, 8, 16, 8192, 512, 512), (16, 8, 64, 16384, 512, 512)])
def test_moe_slab_plan_matches_rule(moe_slab_fn, M, topk, E, H, I, SI):
    st, p = moe_slab_fn(M, topk, E, H, I, SI)
    want = moe_slab_rule(M, topk, E, H, I, SI)
    if want is None:
        assert st == 2
        return
    assert st == 0
    got = dict(split=p.split, k_slab=p.k_slab, tiles_per_cta=p.tiles_per_cta, groups=p.groups,
               chunk_pairs=p.chunk_pairs, slab_bytes=p.slab_bytes, stages=p.stages, ctas_per_sm=p.ctas_per_sm,
               smem_bytes=p.smem_bytes)
    assert got == want
    assert p.stage_bytes == 20480 and p.columns == M * topk + -(-M // p.chunk_pairs)
    assert p.tiles == max(I // 64, -(-SI // 64))
    assert (p.split - 1) * p.k_slab < H and p.slab_bytes >= min(M * topk, p.chunk_pairs) * p.k_slab * 2


def test_moe_slab_plan_decode_block(moe_slab_fn):
    # one token of the E = 128, top-8, H = 4096, I = SI = 1536 block: 9 columns
    # x 24 tiles split in two (432 CTAs, one wave at three per SM); 8 tokens
    # (~53 experts): the grouped form, pairs of 2, 12 groups of 2 tiles
    st, p = moe_slab_fn(1, 8, 128, 4096, 1536, 1536)
    assert st == 0 and (p.split, p.k_slab, p.tiles_per_cta, p.columns, p.tiles) == (2, 2048, 0, 9, 24)
    st, p = moe_slab_fn(8, 8, 128, 4096, 1536, 1536)
    assert st == 0 and (p.split, p.tiles_per_cta, p.groups, p.chunk_pairs) == (1, 2, 12, 2)


def test_moe_slab_plan_rejects_bad_arguments(moe_slab_fn):
    assert moe_slab_fn(0, 8, 128, 4096, 1536, 1536)[0] == 1
    assert moe_slab_fn(1, 8, 128, 4096, 1536, 1536, regs=0)[0] == 1
    assert moe_slab_fn(1, 8, 128, 4096, 1536, 1536, sms=0)[0] == 1
    assert moe_slab_fn(1, 8, 128, 4000, 1536, 1536)[0] == 2   # H % 64
    assert moe_slab_fn(200, 8, 128, 4096, 1536, 1536)[0] == 2  # M * topk > 1024
    assert moe_slab_fn(65, 8, 128, 4096, 1536, 1536)[0] == 2   # beyond 64 tokens: the tcgen05 kernel


# --- the slab kernel's MoE down_combine plan, host only -----------------------------------

class MoeDownSlabPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("tiles_per_cta", "groups", "columns", "chunk_pairs", "slab_bytes",
                                            "stage_bytes", "stages", "ctas_per_sm", "persistent")] + \
        [("smem_bytes", ctypes.c_size_t)]


@pytest.fixture(scope="module")
def down_slab_fn():
    from moe_nvfp4_gemv_gb300 import fp4gemv
    f = fp4gemv.lib().fp4gemv_plan_moe_down_slab
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 8 + [ctypes.POINTER(MoeDownSlabPlan)]

    def plan(M, topk, E, H, I, SI, regs=128, sms=SMS):
        out = MoeDownSlabPlan()
        return f(M, topk, E, H, I, SI, sms, regs, ctypes.byref(out)), out
    return plan


def down_slab_rule(M, topk, E, H, I, SI, sms=SMS):
    """The rule written out: 1 <= M <= 64; chunks of 8 pairs (rows
    min(P, 8) of max(I, SI) bf16).  Expected streaming columns C: the
    expected distinct experts of P uniform draws (at least ceil(P / 8)
    chunks) plus ceil(M / 8) shared-expert chunks; n(T) = C ceil(tiles / T).
    One tile at two CTAs per SM when n(1) fits one wave of two per SM, two
    tiles at two per SM when n(2) does, one tile at three per SM when n(2)
    fills more than 0.9 and at most 1.35 waves of three per SM, else two
    tiles at three per SM.  When that grid holds more than one wave (n(T) >
    occ x sms): the persistent grid at three per SM, chunks of 4 pairs if
    P <= E (C and n recomputed with them), T = 4 if n(4) is at least
    1.6 x 3 sms, else 2 if n(2) is, else 1.  As many 18 KB stages as
    fit beside the slab within 228 KB / occ less 4 KB (2 .. 8; on the grid
    form at most T stage streams of I).  The reported T is the largest
    group, ceil(tiles / groups)."""
    if M < 1 or M > 64:
        return None
    P = M * topk
    tiles = -(-H // 128)
    cols = max(E * (1.0 - (1.0 - 1.0 / E) ** P), float(-(-P // 8))) + -(-M // 8)
    n = lambda T: cols * -(-tiles // T)  # noqa: E731
    f = n(2) / (3.0 * sms)
    if n(1) <= 2.0 * sms:
        T, occ = 1, 2
    elif n(2) <= 2.0 * sms:
        T, occ = 2, 2
    elif 0.9 < f <= 1.35:
        T, occ = 1, 3
    else:
        T, occ = 2, 3
    persistent = n(T) > occ * sms
    chunk = 8
    if persistent:
        occ = 3
        if P <= E:
            chunk = 4
            cols = max(E * (1.0 - (1.0 - 1.0 / E) ** P), float(-(-P // 4))) + -(-M // 4)
        T = 4 if n(4) >= 1.6 * 3 * sms else 2 if n(2) >= 1.6 * 3 * sms else 1
    rows = min(P, chunk)
    nst = -(-max(I, SI) // 256)
    slab = -(-(rows * nst * 512) // 1024) * 1024
    ns = min(8, (228 * 1024 // occ - 4096 - 1024 - slab) // 18432)
    if not persistent:
        ns = min(ns, T * -(-I // 256))
    if ns < 2:
        return None
    groups = -(-tiles // T)
    return dict(tiles_per_cta=-(-tiles // groups), groups=groups, chunk_pairs=chunk, slab_bytes=slab, stages=ns,
                ctas_per_sm=occ, persistent=int(persistent), smem_bytes=1024 + slab + ns * 18432)


def test_moe_slab_rule_decode_block():
    # gate_up of the E = 128, top-8, H = 4096, I = SI = 1536 block on 152
    # SMs: the shapes the sweep found best (split form at one token)
    c = (8, 128, 4096, 1536, 1536)
    got = {M: (moe_slab_rule(M, *c)["split"], moe_slab_rule(M, *c)["tiles_per_cta"], moe_slab_rule(M, *c)["chunk_pairs"],
               moe_slab_rule(M, *c)["ctas_per_sm"]) for M in (1, 2, 3, 4, 5, 6, 7, 8, 9, 32)}
    assert got == {1: (2, 0, 4, 3), 2: (1, 1, 1, 3), 3: (1, 2, 4, 2), 4: (1, 2, 2, 3), 5: (1, 1, 2, 3), 6: (1, 1, 2, 3),
                   7: (1, 1, 2, 3), 8: (1, 2, 2, 3), 9: (1, 2, 2, 3), 32: (1, 2, 4, 2)}


def test_down_slab_rule_decode_block():
    # the E = 128, top-8, H = 4096, I = SI = 1536 block on 152 SMs: the
    # shapes the sweep found best at 1, 2, 4 and 8 tokens
    c = (8, 128, 4096, 1536, 1536)
    got = {M: tuple(down_slab_rule(M, *c)[k] for k in ("tiles_per_cta", "ctas_per_sm", "persistent"))
           for M in (1, 2, 3, 4, 5, 6, 8, 16, 32, 64)}
    assert got == {1: (1, 2, 0), 2: (2, 2, 0), 3: (2, 3, 0), 4: (1, 3, 1), 5: (1, 3, 1), 6: (1, 3, 1), 8: (2, 3, 1),
                   16: (2, 3, 1), 32: (4, 3, 1), 64: (4, 3, 1)}


@pytest.mark.parametrize("M,topk,E,H,I,SI", [(1, 8, 128, 4096, 1536, 1536), (8, 8, 128, 4096, 1536, 1536),
                                             (32, 8, 128, 4096, 1536, 1536), (64, 8, 128, 4096, 1536, 1536),
                                             (16, 8, 128, 832, 256, 256), (3, 2, 8, 384, 256, 512),
                                             (20, 2, 8, 384, 256, 512), (1, 8, 300, 4096, 1536, 1536),
                                             (4, 8, 128, 4096, 8192, 1536), (65, 8, 128, 4096, 1536, 1536),
                                             (64, 8, 16, 4096, 16384, 1536)])
def test_down_slab_plan_matches_rule(down_slab_fn, M, topk, E, H, I, SI):
    st, p = down_slab_fn(M, topk, E, H, I, SI)
    want = down_slab_rule(M, topk, E, H, I, SI)
    if want is None:
        assert st == 2
        return
    assert st == 0
    got = dict(tiles_per_cta=p.tiles_per_cta, groups=p.groups, chunk_pairs=p.chunk_pairs, slab_bytes=p.slab_bytes,
               stages=p.stages, ctas_per_sm=p.ctas_per_sm, persistent=p.persistent, smem_bytes=p.smem_bytes)
    assert got == want
    assert p.stage_bytes == 18432 and p.columns == M * topk + -(-M // p.chunk_pairs)
    # the groups split the tiles evenly: floor or ceil of tiles / groups each
    tiles = -(-H // 128)
    sizes = [(g + 1) * tiles // p.groups - g * tiles // p.groups for g in range(p.groups)]
    assert sum(sizes) == tiles and max(sizes) == p.tiles_per_cta and max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("topk,E,H,I,SI", [(8, 128, 4096, 1536, 1536), (8, 256, 7168, 2048, 2048),
                                           (2, 8, 4096, 14336, 14336), (4, 64, 2048, 768, 1536)])
def test_down_slab_plan_matches_rule_every_m(down_slab_fn, topk, E, H, I, SI):
    # every token count 1 .. 64 (grid form, persistent form and the switch
    # between them, chunks of 4 or 8), and no plan past 64 tokens
    for M in range(1, 66):
        st, p = down_slab_fn(M, topk, E, H, I, SI)
        want = down_slab_rule(M, topk, E, H, I, SI)
        if want is None:
            assert st == 2, M
            continue
        assert st == 0, M
        got = dict(tiles_per_cta=p.tiles_per_cta, groups=p.groups, chunk_pairs=p.chunk_pairs,
                   slab_bytes=p.slab_bytes, stages=p.stages, ctas_per_sm=p.ctas_per_sm, persistent=p.persistent,
                   smem_bytes=p.smem_bytes)
        assert got == want, M


def test_down_slab_plan_decode_block(down_slab_fn):
    # E = 128, top-8, H = 4096, I = SI = 1536: one token, one tile per CTA at
    # two CTAs per SM (its 288 CTAs in one wave); 8 tokens, the persistent
    # grid at three per SM, chunks of 4 pairs (64 pairs over 128 experts),
    # items of two tiles; 32 tokens, chunks of 8 pairs and items of four
    st, p = down_slab_fn(1, 8, 128, 4096, 1536, 1536)
    assert st == 0 and (p.tiles_per_cta, p.groups, p.chunk_pairs, p.ctas_per_sm, p.persistent) == (1, 32, 8, 2, 0)
    st, p = down_slab_fn(8, 8, 128, 4096, 1536, 1536)
    assert st == 0 and (p.tiles_per_cta, p.groups, p.chunk_pairs, p.ctas_per_sm, p.persistent) == (2, 16, 4, 3, 1)
    st, p = down_slab_fn(32, 8, 128, 4096, 1536, 1536)
    assert st == 0 and (p.tiles_per_cta, p.groups, p.chunk_pairs, p.ctas_per_sm, p.persistent) == (4, 8, 8, 3, 1)


def test_down_slab_plan_rejects_bad_arguments(down_slab_fn):
    assert down_slab_fn(0, 8, 128, 4096, 1536, 1536)[0] == 1
    assert down_slab_fn(1, 8, 128, 4096, 1536, 1536, regs=0)[0] == 1
    assert down_slab_fn(1, 8, 128, 4096, 1536, 1536, sms=0)[0] == 1
    assert down_slab_fn(1, 8, 128, 4096, 192, 1536)[0] == 2   # I < 256
