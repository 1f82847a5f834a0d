"""GPU parity of the MoE pair (gate_up, down_combine) against the FP64
oracle, plus an exact-integer routing probe, duplicate experts, expert
chunks larger than one token tile, and out-of-range ids."""
import numpy as np
import pytest
import torch

import oracle
from moe_nvfp4_gemv_gb300 import synth
from gpu_util import assert_close, require_gpu, u16

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def fp4():
    require_gpu()
    from moe_nvfp4_gemv_gb300 import fp4gemv
    return fp4gemv


def make_moe(M, E, H, I, SI, topk, seed=0, ids=None):
    if ids is None:
        ids, tw = synth.routing(M, E, topk, seed=seed)
    else:
        tw = torch.softmax(torch.randn(M, topk, generator=torch.Generator().manual_seed(seed)), dim=1)
    d = dict(M=M, E=E, H=H, I=I, SI=SI, topk=topk, ids=ids.to(torch.int32).contiguous(), tw=tw.float().contiguous())
    d["x"] = synth.activations(M, H, seed=seed + 1)
    d["w1"] = torch.stack([synth.fp4_bytes(2 * I, H, seed=seed + 100 + e) for e in range(E)])
    d["w1_sf"] = torch.cat([synth.e4m3_bytes(oracle.scale_bytes(2 * I, H), seed=seed + 300 + e) for e in range(E)])
    d["alpha"] = synth.expert_alphas(E)
    d["wsh"] = synth.fp4_bytes(2 * SI, H, seed=seed + 2)
    d["ssh"] = synth.e4m3_bytes(oracle.scale_bytes(2 * SI, H), seed=seed + 3)
    d["gssh"] = torch.tensor([0.01])
    d["act"] = synth.activations(M * topk, I, seed=seed + 4)
    d["sact"] = synth.activations(M, SI, seed=seed + 5)
    d["w2"] = torch.stack([synth.fp4_bytes(H, I, seed=seed + 500 + e) for e in range(E)])
    d["w2_sf"] = torch.cat([synth.e4m3_bytes(oracle.scale_bytes(H, I), seed=seed + 700 + e) for e in range(E)])
    d["alpha2"] = synth.expert_alphas(E)
    d["wsd"] = synth.fp4_bytes(H, SI, seed=seed + 6)
    d["ssd"] = synth.e4m3_bytes(oracle.scale_bytes(H, SI), seed=seed + 7)
    d["gssd"] = torch.tensor([0.01])
    return d


def run_gate_up(fp4, d, pdl=True):
    g = {k: v.to(DEV) for k, v in d.items() if isinstance(v, torch.Tensor)}
    act = torch.full((d["M"] * d["topk"], d["I"]), 7.0, dtype=torch.bfloat16, device=DEV)
    sact = torch.full((d["M"], d["SI"]), 7.0, dtype=torch.bfloat16, device=DEV)
    fp4.moe_gate_up(g["x"], g["ids"], g["w1"], g["w1_sf"], g["alpha"], act, g["wsh"], g["ssh"], g["gssh"], sact, pdl=pdl)
    return act, sact


def run_down(fp4, d, pdl=True):
    g = {k: v.to(DEV) for k, v in d.items() if isinstance(v, torch.Tensor)}
    out = torch.full((d["M"], d["H"]), 7.0, dtype=torch.bfloat16, device=DEV)
    fp4.moe_down_combine(g["act"], g["ids"], g["tw"], g["w2"], g["w2_sf"], g["alpha2"], g["sact"], g["wsd"], g["ssd"],
                         g["gssd"], out, pdl=pdl)
    return out


def ref_gate_up(d, pairs=None, tokens=None):
    return oracle.moe_gate_up(u16(d["x"]), d["ids"].numpy(), d["w1"].numpy(), d["w1_sf"].numpy(), d["alpha"].numpy(),
                              d["wsh"].numpy(), d["ssh"].numpy(), float(d["gssh"][0]), pairs=pairs, tokens=tokens)


def ref_down(d, tokens=None):
    return oracle.moe_down_combine(u16(d["act"]), d["ids"].numpy(), d["tw"].numpy(), d["w2"].numpy(),
                                   d["w2_sf"].numpy(), d["alpha2"].numpy(), u16(d["sact"]), d["wsd"].numpy(),
                                   d["ssd"].numpy(), float(d["gssd"][0]), tokens=tokens)


@pytest.mark.parametrize("M", [1, 3, 16, 20])
def test_gate_up_small(fp4, M):
    d = make_moe(M, E=8, H=512, I=256, SI=384, topk=2, seed=M)
    act, sact = run_gate_up(fp4, d)
    (an, al, ah), (sn, sl, sh), bad = ref_gate_up(d)
    assert bad == 0
    assert_close(u16(act), (an, al, ah), f"act M={M}")
    assert_close(u16(sact), (sn, sl, sh), f"sact M={M}")
    assert fp4.get_device_error() == 0


@pytest.mark.parametrize("M", [1, 3, 16, 20])
def test_down_combine_small(fp4, M):
    d = make_moe(M, E=8, H=384, I=256, SI=512, topk=2, seed=50 + M)
    out = run_down(fp4, d)
    ref, bad = ref_down(d)
    assert bad == 0
    assert_close(u16(out), ref, f"down M={M}")
    assert fp4.get_device_error() == 0


# Above 64 tokens both MoE kernels run on the tcgen05 path (chunks of up to
# 32 pairs per expert); with 4 experts and top-2 each expert gets several
# chunks and a ragged last one.
@pytest.mark.parametrize("M", [72, 130])
def test_gate_up_tcgen05_path(fp4, M):
    d = make_moe(M, E=4, H=512, I=256, SI=384, topk=2, seed=300 + M)
    act, sact = run_gate_up(fp4, d)
    (an, al, ah), (sn, sl, sh), bad = ref_gate_up(d)
    assert bad == 0
    assert_close(u16(act), (an, al, ah), f"act M={M}")
    assert_close(u16(sact), (sn, sl, sh), f"sact M={M}")
    assert fp4.get_device_error() == 0


@pytest.mark.parametrize("M", [72, 130])
def test_down_combine_tcgen05_path(fp4, M):
    d = make_moe(M, E=4, H=384, I=512, SI=256, topk=2, seed=400 + M)
    out = run_down(fp4, d)
    ref, bad = ref_down(d)
    assert bad == 0
    assert_close(u16(out), ref, f"down M={M}")
    assert fp4.get_device_error() == 0


def _random_moe_cases(n=8, seed=77):
    """Seeded random MoE layers: tokens alternate between the register-fed
    range (<= 64) and the tcgen05 range (> 64); E, top-k and the widths vary
    (multiples of 64, at least 256 where the kernels require it)."""
    rng = np.random.RandomState(seed)
    cases = []
    for i in range(n):
        M = int(rng.randint(1, 65)) if i % 2 == 0 else int(rng.randint(65, 161))
        E = int(rng.randint(2, 17))
        topk = int(rng.randint(1, min(E, 4) + 1))
        H, I, SI = (64 * int(rng.randint(4, 13)) for _ in range(3))
        cases.append((M, E, topk, H, I, SI))
    return cases


@pytest.mark.parametrize("M,E,topk,H,I,SI", _random_moe_cases())
def test_moe_random_shapes(fp4, M, E, topk, H, I, SI):
    d = make_moe(M, E=E, H=H, I=I, SI=SI, topk=topk, seed=M * 31 + E)
    act, sact = run_gate_up(fp4, d)
    (an, al, ah), (sn, sl, sh), bad = ref_gate_up(d)
    assert bad == 0
    assert_close(u16(act), (an, al, ah), f"act M={M} E={E} topk={topk} H={H} I={I} SI={SI}")
    assert_close(u16(sact), (sn, sl, sh), f"sact M={M} E={E} topk={topk} H={H} I={I} SI={SI}")
    out = run_down(fp4, d)
    ref, bad = ref_down(d)
    assert bad == 0
    assert_close(u16(out), ref, f"down M={M} E={E} topk={topk} H={H} I={I} SI={SI}")
    assert fp4.get_device_error() == 0


def test_repeated_and_crowded_experts(fp4):
    # every token routes both slots to expert 3 (a repeated expert within a
    # token) and 40 tokens share it: its pair list spans several token tiles.
    M, topk = 40, 2
    ids = torch.full((M, topk), 3, dtype=torch.int32)
    ids[::5, 1] = 1
    d = make_moe(M, E=4, H=256, I=256, SI=256, topk=topk, seed=9, ids=ids)
    act, sact = run_gate_up(fp4, d)
    (an, al, ah), (sn, sl, sh), _ = ref_gate_up(d)
    assert_close(u16(act), (an, al, ah), "act crowded")
    assert_close(u16(sact), (sn, sl, sh), "sact crowded")
    out = run_down(fp4, d)
    ref, _ = ref_down(d)
    assert_close(u16(out), ref, "down crowded")


def test_routing_probe_exact(fp4):
    # W2[e] is 1.0 in K column 0 with block-0 scale 2^e, act rows one-hot at
    # column 0, tw = [1, 1/16], alpha2 = 1, zero shared expert:
    # out[t, h] = 2^e0 + 2^(e1-4) exactly.
    M, E, H, I, SI, topk = 6, 4, 256, 256, 256, 2
    w2 = torch.zeros(E, H, I // 2, dtype=torch.uint8)
    w2[:, :, 0] = 0x02
    sfe = oracle.scale_bytes(H, I)
    w2_sf = np.full(E * sfe, 0x38, np.uint8)
    for e in range(E):
        for h in range(H):
            w2_sf[e * sfe + oracle.swz(h, 0, I)] = 0x38 + 8 * e
    ids = torch.tensor([[0, 1], [3, 2], [2, 0], [1, 3], [3, 0], [2, 1]], dtype=torch.int32)
    act = torch.zeros(M * topk, I, dtype=torch.bfloat16)
    act[:, 0] = 1.0
    d = dict(M=M, H=H, act=act.to(DEV), ids=ids.to(DEV), tw=torch.tensor([[1.0, 1 / 16]] * M).to(DEV),
             w2=w2.to(DEV), w2_sf=torch.from_numpy(w2_sf).to(DEV), alpha2=torch.ones(E, device=DEV),
             sact=torch.zeros(M, SI, dtype=torch.bfloat16, device=DEV),
             wsd=torch.zeros(H, SI // 2, dtype=torch.uint8, device=DEV),
             ssd=torch.zeros(oracle.scale_bytes(H, SI), dtype=torch.uint8, device=DEV),
             gssd=torch.ones(1, device=DEV))
    out = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
    fp4.moe_down_combine(d["act"], d["ids"], d["tw"], d["w2"], d["w2_sf"], d["alpha2"], d["sact"], d["wsd"], d["ssd"],
                         d["gssd"], out)
    want = torch.tensor([2.0 ** int(a) + 2.0 ** (int(b) - 4) for a, b in ids.tolist()])
    assert torch.equal(out.float().cpu(), want[:, None].expand(M, H))


def test_bad_expert_id_reported(fp4):
    d = make_moe(3, E=4, H=256, I=256, SI=256, topk=2, seed=21)
    d["ids"][1, 1] = 17
    act, _ = run_gate_up(fp4, d)
    assert fp4.get_device_error() == 6
    rows = [0, 1, 2, 4, 5]
    (an, al, ah), _, _ = ref_gate_up(d, pairs=rows)
    assert_close(u16(act)[rows], (an[rows], al[rows], ah[rows]), "act with a bad id elsewhere")
    assert (act[3] == 7.0).all()  # the bad pair's row is left unwritten
    out = run_down(fp4, d)
    assert fp4.get_device_error() == 6
    ref, _ = ref_down(d, tokens=[0, 2])
    assert_close(u16(out)[[0, 2]], tuple(r[[0, 2]] for r in ref), "down with a bad id elsewhere")
    assert (out[1] == 7.0).all()  # the token with the bad id is left unwritten
    assert fp4.get_device_error() == 0


@pytest.mark.parametrize("M", list(synth.MOE_M))
def test_moe_config(fp4, M):
    c = synth.MOE
    d = make_moe(M, c["E"], c["H"], c["I"], c["SI"], c["topk"], seed=100)
    act, sact = run_gate_up(fp4, d)
    P = M * c["topk"]
    pairs = list(range(P)) if P <= 64 else sorted(set(np.random.default_rng(M).integers(0, P, 24).tolist()) | {0, P - 1})
    tokens = list(range(M)) if M <= 8 else [0, M // 2, M - 1]
    (an, al, ah), (sn, sl, sh), bad = ref_gate_up(d, pairs=pairs, tokens=tokens)
    assert bad == 0
    assert_close(u16(act)[pairs], (an[pairs], al[pairs], ah[pairs]), f"act M={M}")
    assert_close(u16(sact)[tokens], (sn[tokens], sl[tokens], sh[tokens]), f"sact M={M}")
    out = run_down(fp4, d)
    ref, bad = ref_down(d, tokens=tokens)
    assert_close(u16(out)[tokens], tuple(r[tokens] for r in ref), f"down M={M}")
    assert fp4.get_device_error() == 0


def test_workspace_reuse_across_shapes(fp4):
    # one uninitialised workspace (sized for the largest call) serves calls of
    # different M and H in turn, on the grid and the persistent form (E = 128):
    # nothing is carried between calls
    c = synth.MOE
    ws = torch.full((fp4.moe_down_combine_workspace_bytes(32, c["topk"], 1024),), 0xA5, dtype=torch.uint8,
                    device=DEV)
    for M, H, E in ((5, 1024, 16), (32, 256, 16), (32, 1024, 128), (1, 1024, 16), (17, 512, 16), (32, 1024, 128),
                    (32, 1024, 16)):
        d = make_moe(M, E, H, 512, 512, c["topk"], seed=M + E)
        g = {k: v.to(DEV) for k, v in d.items() if isinstance(v, torch.Tensor)}
        out = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
        fp4.moe_down_combine(g["act"], g["ids"], g["tw"], g["w2"], g["w2_sf"], g["alpha2"], g["sact"], g["wsd"],
                             g["ssd"], g["gssd"], out, workspace=ws)
        ref, _ = ref_down(d)
        assert_close(u16(out), ref, f"workspace reuse M={M}")


def _moe_slab_plan(fp4, M, topk, E, H, I, SI):
    """The slab kernel's gate_up plan for this call on this GPU as (split,
    tiles per CTA; 0 in the split form), or None when the call runs on
    another kernel."""
    import ctypes

    class Plan(ctypes.Structure):
        _fields_ = [(n, ctypes.c_int) for n in ("split", "k_slab", "tiles_per_cta", "groups", "chunk_pairs",
                                                "columns", "tiles", "slab_bytes", "stage_bytes", "stages",
                                                "ctas_per_sm")] + [("smem_bytes", ctypes.c_size_t)]
    f = fp4.lib().fp4gemv_plan_moe_slab
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 8 + [ctypes.POINTER(Plan)]
    out = Plan()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return (out.split, out.tiles_per_cta) if f(M, topk, E, H, I, SI, sms, 125, ctypes.byref(out)) == 0 else None


def _moe_slab_split(fp4, M, topk, E, H, I, SI):
    """Split of the slab kernel's split-form plan (None otherwise)."""
    plan = _moe_slab_plan(fp4, M, topk, E, H, I, SI)
    return plan[0] if plan is not None and plan[1] == 0 else None


# gate_up on the slab kernel (routed chunks of up to 4 pairs of one expert,
# H split over clusters of 1, 2, 4 and 8 CTAs): both outputs element by
# element against the oracle.
@pytest.mark.parametrize("M,topk,E,H,split", [(1, 2, 8, 256, 1), (1, 4, 8, 512, 2), (2, 2, 8, 1024, 4),
                                              (3, 2, 8, 2048, 8), (1, 8, 16, 4096, 8)])
def test_gate_up_slab_splits(fp4, M, topk, E, H, split):
    I, SI = 192, 320
    assert _moe_slab_split(fp4, M, topk, E, H, I, SI) == split
    d = make_moe(M, E=E, H=H, I=I, SI=SI, topk=topk, seed=600 + H + M)
    act, sact = run_gate_up(fp4, d)
    (an, al, ah), (sn, sl, sh), bad = ref_gate_up(d)
    assert bad == 0
    assert_close(u16(act), (an, al, ah), f"act slab M={M} H={H}")
    assert_close(u16(sact), (sn, sl, sh), f"sact slab M={M} H={H}")
    assert fp4.get_device_error() == 0


# Repeated experts on the slab kernel: 8 pairs of one expert (two full
# chunks), and a token that sends 5 of its 8 slots to one expert (a full
# chunk and a ragged one) and 3 to another.
@pytest.mark.parametrize("M,topk,ids", [(2, 4, [[2, 2, 2, 2], [2, 2, 2, 2]]),
                                        (1, 8, [[5, 1, 5, 1, 1, 5, 1, 1]])])
def test_gate_up_slab_repeated_experts(fp4, M, topk, ids):
    E, H, I, SI = 8, 1024, 256, 256
    assert _moe_slab_split(fp4, M, topk, E, H, I, SI) is not None
    d = make_moe(M, E=E, H=H, I=I, SI=SI, topk=topk, seed=31, ids=torch.tensor(ids, dtype=torch.int32))
    act, sact = run_gate_up(fp4, d)
    (an, al, ah), (sn, sl, sh), _ = ref_gate_up(d)
    assert_close(u16(act), (an, al, ah), "act slab repeated")
    assert_close(u16(sact), (sn, sl, sh), "sact slab repeated")
    assert fp4.get_device_error() == 0


def test_gate_up_slab_decode_block(fp4):
    # one token of the E = 128, top-8, H = 4096, I = SI = 1536 block takes the
    # slab kernel with a split of two; every output against the oracle, and
    # two calls in a row agree bit for bit
    c = synth.MOE
    assert _moe_slab_split(fp4, 1, c["topk"], c["E"], c["H"], c["I"], c["SI"]) == 2
    d = make_moe(1, c["E"], c["H"], c["I"], c["SI"], c["topk"], seed=7)
    act, sact = run_gate_up(fp4, d)
    act2, sact2 = run_gate_up(fp4, d)
    assert torch.equal(act, act2) and torch.equal(sact, sact2)
    (an, al, ah), (sn, sl, sh), bad = ref_gate_up(d)
    assert bad == 0
    assert_close(u16(act), (an, al, ah), "act decode block M=1")
    assert_close(u16(sact), (sn, sl, sh), "sact decode block M=1")
    assert fp4.get_device_error() == 0


def _down_slab_plan(fp4, M, topk, E, H, I, SI):
    """The slab plan for this down_combine call on this GPU (None: another
    kernel serves it)."""
    import ctypes

    class Plan(ctypes.Structure):
        _fields_ = [(n, ctypes.c_int) for n in ("tiles_per_cta", "groups", "columns", "chunk_pairs", "slab_bytes",
                                                "stage_bytes", "stages", "ctas_per_sm", "persistent")] + \
            [("smem_bytes", ctypes.c_size_t)]
    f = fp4.lib().fp4gemv_plan_moe_down_slab
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 8 + [ctypes.POINTER(Plan)]
    out = Plan()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return out if f(M, topk, E, H, I, SI, sms, 128, ctypes.byref(out)) == 0 else None


def _down_slab_tiles(fp4, M, topk, E, H, I, SI):
    """Row tiles per CTA (or per item of the persistent grid) of the slab
    plan for this down_combine call on this GPU (None: another kernel serves
    it)."""
    p = _down_slab_plan(fp4, M, topk, E, H, I, SI)
    return None if p is None else p.tiles_per_cta


# down_combine on the slab kernel with two row tiles per CTA: H = 832 is
# 6.5 tiles (a partial last tile, and a last group of one tile); many
# experts, so many columns are inactive duplicates that leave at once and
# the combine waits only for the CTAs that compute.
@pytest.mark.parametrize("M,topk,E,H,I,SI,T", [(16, 8, 128, 832, 256, 256, 2), (12, 8, 96, 1024, 320, 448, 2)])
def test_down_combine_slab_tiles(fp4, M, topk, E, H, I, SI, T):
    assert _down_slab_tiles(fp4, M, topk, E, H, I, SI) == T
    d = make_moe(M, E=E, H=H, I=I, SI=SI, topk=topk, seed=800 + M)
    out = run_down(fp4, d)
    ref, bad = ref_down(d)
    assert bad == 0
    assert_close(u16(out), ref, f"down slab M={M} H={H}")
    assert fp4.get_device_error() == 0
    out2 = run_down(fp4, d)
    assert torch.equal(out, out2)


def test_down_combine_slab_decode_block(fp4):
    # 8 tokens of the E = 128, top-8, H = 4096, I = SI = 1536 block: two row
    # tiles per CTA; sampled tokens against the oracle
    c = synth.MOE
    assert _down_slab_tiles(fp4, 8, c["topk"], c["E"], c["H"], c["I"], c["SI"]) == 2
    d = make_moe(8, c["E"], c["H"], c["I"], c["SI"], c["topk"], seed=101)
    out = run_down(fp4, d)
    tokens = [0, 3, 7]
    ref, bad = ref_down(d, tokens=tokens)
    assert bad == 0
    assert_close(u16(out)[tokens], tuple(r[tokens] for r in ref), "down slab decode block M=8")
    assert fp4.get_device_error() == 0


# The persistent grid (more items than one wave of CTAs): three CTAs per SM
# take (tile group, column) items from a counter.  32 tokens of the decode
# block: groups of 4 tiles; 64 tokens over 1024 experts with H = 832: two
# groups of 3 and 4 tiles, one partial; 32 tokens with H = 1024: one tile per
# item.  Each call twice on one workspace (the counter of the first call is
# stale for the second), sampled or whole outputs against the oracle.
@pytest.mark.parametrize("M,topk,E,H,I,SI,T", [(32, 8, 128, 4096, 1536, 1536, 4), (64, 8, 1024, 832, 256, 256, 4),
                                               (32, 8, 128, 1024, 512, 512, 1)])
def test_down_combine_persistent(fp4, M, topk, E, H, I, SI, T):
    p = _down_slab_plan(fp4, M, topk, E, H, I, SI)
    assert p is not None and p.persistent == 1 and p.tiles_per_cta == T
    d = make_moe(M, E=E, H=H, I=I, SI=SI, topk=topk, seed=1300 + M + E)
    g = {k: v.to(DEV) for k, v in d.items() if isinstance(v, torch.Tensor)}
    ws = torch.full((fp4.moe_down_combine_workspace_bytes(M, topk, H),), 0xA5, dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(2):
        out = torch.full((M, H), 7.0, dtype=torch.bfloat16, device=DEV)
        fp4.moe_down_combine(g["act"], g["ids"], g["tw"], g["w2"], g["w2_sf"], g["alpha2"], g["sact"], g["wsd"],
                             g["ssd"], g["gssd"], out, workspace=ws)
        outs.append(out)
    assert fp4.get_device_error() == 0
    tokens = list(range(M)) if H * I <= 1 << 20 else [0, 5, M // 2, M - 1]
    ref, bad = ref_down(d, tokens=tokens)
    assert bad == 0
    assert_close(u16(outs[0])[tokens], tuple(r[tokens] for r in ref), f"down persistent M={M} E={E} H={H}")
    assert torch.equal(outs[0], outs[1])


def test_down_combine_persistent_crowded_experts(fp4):
    # The persistent grid's plan assumes uniform routing; here 32 tokens send
    # their 8 pairs to 12 of 128 experts (each of those gets ~21 pairs: two
    # or three full chunks of 8), so items of 8 activation rows and experts
    # split over several columns meet most columns being inactive duplicates.
    M, topk, E, H, I, SI = 32, 8, 128, 1024, 512, 512
    p = _down_slab_plan(fp4, M, topk, E, H, I, SI)
    assert p is not None and p.persistent == 1
    g = torch.Generator().manual_seed(5)
    hot = torch.randperm(E, generator=g)[:12]
    ids = torch.stack([hot[torch.randperm(12, generator=g)[:topk]] for _ in range(M)])
    d = make_moe(M, E=E, H=H, I=I, SI=SI, topk=topk, seed=1400, ids=ids)
    out = run_down(fp4, d)
    ref, bad = ref_down(d)
    assert bad == 0
    assert_close(u16(out), ref, "down persistent crowded")
    assert fp4.get_device_error() == 0


def test_down_combine_slab_decode_block_one_token(fp4):
    # one token of the E = 128, top-8, H = 4096, I = SI = 1536 block: one row
    # tile per CTA at two CTAs per SM (288 CTAs, one wave), then the combine
    # kernel; the whole output against the oracle
    c = synth.MOE
    assert _down_slab_tiles(fp4, 1, c["topk"], c["E"], c["H"], c["I"], c["SI"]) == 1
    d = make_moe(1, c["E"], c["H"], c["I"], c["SI"], c["topk"], seed=102)
    out = run_down(fp4, d)
    ref, bad = ref_down(d)
    assert bad == 0
    assert_close(u16(out), ref, "down slab decode block M=1")
    assert fp4.get_device_error() == 0


# More experts per token than one group of the combine's loads (8), and a
# single expert per token: gate_up and down_combine (slab kernel, then the
# combine kernel) against the oracle.
@pytest.mark.parametrize("M,topk", [(3, 12), (20, 12), (2, 1)])
def test_moe_topk_beyond_one_load_group(fp4, M, topk):
    E, H, I, SI = 32, 384, 512, 256
    d = make_moe(M, E=E, H=H, I=I, SI=SI, topk=topk, seed=1200 + M + topk)
    act, sact = run_gate_up(fp4, d)
    (an, al, ah), (sn, sl, sh), bad = ref_gate_up(d)
    assert bad == 0
    assert_close(u16(act), (an, al, ah), f"act M={M} topk={topk}")
    assert_close(u16(sact), (sn, sl, sh), f"sact M={M} topk={topk}")
    out = run_down(fp4, d)
    ref, bad = ref_down(d)
    assert bad == 0
    assert_close(u16(out), ref, f"down M={M} topk={topk}")
    assert fp4.get_device_error() == 0


# I = 256, a single 256-K stage: the slab kernel has no plan (its ring would
# hold fewer than two stages), so down_combine runs on the register-fed
# kernel with its in-kernel arrival counters and combine (one token: the
# converter-warp variant; 8 tokens: the variant budgeted for three CTAs per
# SM).  Then 300 experts on the slab kernel (no per-CTA expert table).
@pytest.mark.parametrize("M", [1, 8])
def test_down_combine_register_fed_path(fp4, M):
    E = 300
    assert _down_slab_tiles(fp4, M, 2, E, 256, 256, 256) is None
    d = make_moe(M, E=E, H=256, I=256, SI=256, topk=2, seed=1000 + M)
    out = run_down(fp4, d)
    ref, bad = ref_down(d)
    assert bad == 0
    assert_close(u16(out), ref, f"down register-fed M={M} E={E}")
    assert fp4.get_device_error() == 0


@pytest.mark.parametrize("M", [1, 8])
def test_down_combine_slab_many_experts(fp4, M):
    E = 300
    assert _down_slab_tiles(fp4, M, 2, E, 256, 512, 256) is not None
    d = make_moe(M, E=E, H=256, I=512, SI=256, topk=2, seed=1100 + M)
    out = run_down(fp4, d)
    ref, bad = ref_down(d)
    assert bad == 0
    assert_close(u16(out), ref, f"down slab M={M} E={E}")
    assert fp4.get_device_error() == 0


# gate_up in the grouped form (the whole H per CTA, several tiles per CTA in
# turn): routed and shared tiles split unevenly over the groups, shared-
# expert boxes that alternate between the halves of their 128-row scale
# groups; then crowded experts (8 experts x 4 pairs: chunks of 4).
@pytest.mark.parametrize("M,topk,E,H,I,SI,ids", [
    (6, 8, 64, 512, 1024, 960, None),
    (4, 8, 16, 1024, 2048, 448, [[0, 1, 2, 3, 4, 5, 6, 7]] * 4),
])
def test_gate_up_slab_grouped(fp4, M, topk, E, H, I, SI, ids):
    plan = _moe_slab_plan(fp4, M, topk, E, H, I, SI)
    assert plan is not None and plan[0] == 1 and plan[1] >= 2
    d = make_moe(M, E=E, H=H, I=I, SI=SI, topk=topk, seed=900 + M,
                 ids=None if ids is None else torch.tensor(ids, dtype=torch.int32))
    act, sact = run_gate_up(fp4, d)
    (an, al, ah), (sn, sl, sh), bad = ref_gate_up(d)
    assert bad == 0
    assert_close(u16(act), (an, al, ah), f"act grouped M={M}")
    assert_close(u16(sact), (sn, sl, sh), f"sact grouped M={M}")
    assert fp4.get_device_error() == 0
