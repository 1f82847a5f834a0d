"""FP64 CPU oracle for the NVFP4 small-M GEMV family -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package.  The CUDA library never calls it, and
the two share no code: the arithmetic lives in ``fp4gemv_oracle.c`` (plain C,
double precision, one function per operation the pages define); this module
only marshals numpy arrays and splits row ranges over host threads (ctypes
releases the GIL during each foreign call).

Conventions: bf16 tensors are numpy ``uint16`` bit patterns; weights, scales
are ``uint8``; every result is a triple ``(nominal, lo, hi)`` of bf16 bit
arrays -- ``nominal`` is the pages' formula with exact arithmetic and
round-to-nearest-even at each rounding the pages name; ``[lo, hi]`` is the
hull of the outputs reached when an INTERMEDIATE bf16 rounding the pages
name (G / U before silu_mul; y_j, y_shared and the top-k sum in
down_combine) takes its other neighbour because the exact value lies next to
a rounding midpoint (within 2^-16 relative for the dot products, within the
rigorous fp32 bound for the top-k sum).  Outputs without such an
intermediate (the plain dense GEMV, bf16_gemv, the routed gate_up) always
have lo == hi == nominal.

Sources (title / section): vllm.models.flint.ops.nvfp4_gemv (module docstring,
nvfp4_gemv, bf16_gemv, dequantize_rows), vllm.models.flint.ops.linear
(_swizzled_scale_buffer), vllm.models.flint.ops.moe_gemv (module docstring,
gate_up, down_combine), vllm.model_executor.kernels.linear.nvfp4.flashinfer
(the W4A4 kernels' apply_weights: scaled_fp4_quant, then the NVFP4 GEMM with
alpha; the quantiser's arithmetic is a reading, see ``quantize_act``).

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
(value tables, closed forms, brute force, a library cross-check and
hand-worked golden cases).  The within-chunk byte order of the 128x4 scale
layout is a reading (the pages name the layout and its size only); it is
pinned by bijection, size and chunk-structure invariants, not by a printed
example.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4gemv_oracle.c")
_LIB = os.path.join(_HERE, "libfp4gemv_oracle.so")
_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_dbl = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libfp4gemv_oracle.so`` (gcc, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            sig = {
                "orc_e2m1": (_dbl, [ctypes.c_int]),
                "orc_e4m3": (_dbl, [ctypes.c_int]),
                "orc_bf16_value": (_dbl, [ctypes.c_int]),
                "orc_bf16_rne": (ctypes.c_uint16, [_dbl]),
                "orc_scale_bytes": (_i64, [_i64, _i64]),
                "orc_swz": (_i64, [_i64, _i64, _i64]),
                "orc_unswz": (None, [_i64, _i64, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
                "orc_w1_row": (_i64, [_i64, ctypes.c_int]),
                "orc_dequant_rows": (None, [_vp, _vp, _i64, _i64, _i64, _vp, _vp]),
                "orc_round_intermediate": (None, [_dbl, _dbl, ctypes.POINTER(ctypes.c_uint16),
                                                  ctypes.POINTER(ctypes.c_uint16)]),
                "orc_gemv_acc": (None, [_vp, _i64, _i64, _vp, _vp, _i64, _vp, _i64, _vp, _vp]),
                "orc_bf16_gemv_acc": (None, [_vp, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _vp]),
                "orc_dense_epilogue": (None, [_vp, _i64, _i64, _dbl, ctypes.c_int, _vp, _vp, _vp]),
                "orc_moe_gate_up_routed": (ctypes.c_int, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _i64, _i64,
                                                          _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
                "orc_moe_gate_up_shared": (None, [_vp, _i64, _i64, _vp, _vp, _dbl, _i64, _i64, _vp, _vp,
                                                  _vp, _vp, _vp]),
                "orc_moe_down_combine": (ctypes.c_int, [_vp, _vp, _vp, _i64, _vp, _vp, _vp, _i64, _i64, _i64,
                                                        _vp, _vp, _vp, _dbl, _i64, _i64, _i64, _vp, _vp, _vp,
                                                        _vp]),
                "orc_e4m3_encode": (ctypes.c_int, [ctypes.c_float]),
                "orc_e2m1_encode": (ctypes.c_int, [ctypes.c_float]),
                "orc_quantize_act": (None, [_vp, _i64, _i64, _i64, ctypes.c_float, _vp, _vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _threads(threads: int | None) -> int:
    return max(1, threads if threads else (os.cpu_count() or 1))


def _chunks(n: int, parts: int):
    parts = max(1, min(parts, n))
    step = (n + parts - 1) // parts
    return [(a, min(n, a + step)) for a in range(0, n, step)]


def _run(fn, ranges, threads):
    if threads == 1 or len(ranges) == 1:
        return [fn(a, b) for a, b in ranges]
    with ThreadPoolExecutor(threads) as ex:
        return list(ex.map(lambda r: fn(*r), ranges))


# --------------------------------------------------------------------------
# Scalars and layout
# --------------------------------------------------------------------------

def e2m1(code: int) -> float:
    return _load().orc_e2m1(int(code))


def e4m3(byte: int) -> float:
    return _load().orc_e4m3(int(byte))


def bf16_value(bits: int) -> float:
    return _load().orc_bf16_value(int(bits))


def bf16_rne(v: float) -> int:
    return int(_load().orc_bf16_rne(float(v)))


def scale_bytes(rows: int, K: int) -> int:
    return int(_load().orc_scale_bytes(rows, K))


def swz(r: int, kb: int, K: int) -> int:
    return int(_load().orc_swz(r, kb, K))


def unswz(off: int, K: int) -> tuple[int, int]:
    r, kb = _i64(), _i64()
    _load().orc_unswz(off, K, ctypes.byref(r), ctypes.byref(kb))
    return r.value, kb.value


def round_intermediate(v: float, eps: float) -> tuple[int, int]:
    """(nominal, alternative) bf16 bits of an intermediate value v: the
    alternative is the other neighbour when a rounding midpoint lies within
    eps of v, else the nominal rounding again."""
    n, a = ctypes.c_uint16(), ctypes.c_uint16()
    _load().orc_round_intermediate(float(v), float(eps), ctypes.byref(n), ctypes.byref(a))
    return int(n.value), int(a.value)


INTERMEDIATE_REL_WINDOW = 2.0 ** -16


def w1_row(i: int, up: bool) -> int:
    return int(_load().orc_w1_row(i, 1 if up else 0))


def scales_logical(sf: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Logical e4m3 scale bytes [rows, K/16] read out of a flat 128x4 buffer."""
    out = np.empty((rows, K // 16), np.uint8)
    for r in range(rows):
        for kb in range(K // 16):
            out[r, kb] = sf[swz(r, kb, K)]
    return out


# --------------------------------------------------------------------------
# Dense ops
# --------------------------------------------------------------------------

def dequantize_rows(w: np.ndarray, sf: np.ndarray, threads: int | None = None) -> np.ndarray:
    """bf16 [rows, K] = e2m1 * e4m3 exactly (no global scale)."""
    lib = _load()
    rows, K = w.shape[0], w.shape[1] * 2
    w = np.ascontiguousarray(w, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8).reshape(-1)
    out = np.empty((rows, K), np.uint16)
    t = _threads(threads)

    def work(a, b):
        tmp = np.empty(K, np.float64)
        lib.orc_dequant_rows(_p(w), _p(sf), K, a, b, _p(tmp), _p(out))

    _run(work, _chunks(rows, 4 * t), t)
    return out


def _dense(acc_fn, x, K, N, gs, silu_mul, rows, threads):
    lib = _load()
    x = np.ascontiguousarray(x, np.uint16)
    M = x.shape[0]
    if silu_mul:
        outs = np.arange(N // 2, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
        wrows = np.concatenate([outs, outs + N // 2])
    else:
        outs = np.arange(N, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
        wrows = outs
    nr = wrows.size
    acc = np.empty((M, nr), np.float64)
    t = _threads(threads)

    def work(a, b):
        sub = np.ascontiguousarray(wrows[a:b])
        tmp = np.empty(K, np.float64)
        pa = np.empty((M, b - a), np.float64)
        acc_fn(x, sub, tmp, pa)
        acc[:, a:b] = pa

    _run(work, _chunks(nr, 4 * t), t)
    nc = outs.size
    nom, lo, hi = (np.empty((M, nc), np.uint16) for _ in range(3))
    lib.orc_dense_epilogue(_p(acc), M, nr, float(gs), 1 if silu_mul else 0, _p(nom), _p(lo), _p(hi))
    return nom, lo, hi


def dense_acc(x, w, sf, rows=None, threads=None) -> np.ndarray:
    """The exact float64 accumulators acc[m, i] = x[m] . dequant(W)[rows[i]]
    (all rows when ``rows`` is None), before any scale or rounding."""
    lib = _load()
    w = np.ascontiguousarray(w, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8).reshape(-1)
    x = np.ascontiguousarray(x, np.uint16)
    N, K = w.shape[0], w.shape[1] * 2
    M = x.shape[0]
    wrows = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    acc = np.empty((M, wrows.size), np.float64)
    tmp = np.empty(K, np.float64)
    lib.orc_gemv_acc(_p(x), K, M, _p(w), _p(sf), K, _p(wrows), wrows.size, _p(tmp), _p(acc))
    return acc


def nvfp4_gemv(x, w, sf, global_scale: float, silu_mul: bool = False, rows=None, threads=None):
    """out = bf16(f32(x @ dequant(W)^T) * gs); with silu_mul, [M, N/2] of
    bf16(silu(G) * U).  ``rows`` selects output columns (sampling)."""
    lib = _load()
    w = np.ascontiguousarray(w, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8).reshape(-1)
    N, K = w.shape[0], w.shape[1] * 2

    def acc_fn(xx, sub, tmp, pa):
        lib.orc_gemv_acc(_p(xx), K, xx.shape[0], _p(w), _p(sf), K, _p(sub), sub.size, _p(tmp), _p(pa))

    return _dense(acc_fn, x, K, N, global_scale, silu_mul, rows, threads)


def bf16_gemv(x, w, silu_mul: bool = False, rows=None, threads=None, global_scale: float = 1.0):
    """BF16-weight variant: W is bf16 [N, K] (uint16 bits), global scale 1
    unless given (the dequantize + GEMM path passes the layer's scale)."""
    lib = _load()
    w = np.ascontiguousarray(w, np.uint16)
    N, K = w.shape

    def acc_fn(xx, sub, tmp, pa):
        lib.orc_bf16_gemv_acc(_p(xx), K, xx.shape[0], _p(w), K, _p(sub), sub.size, _p(tmp), _p(pa))

    return _dense(acc_fn, x, K, N, global_scale, silu_mul, rows, threads)


# --------------------------------------------------------------------------
# MoE pair
# --------------------------------------------------------------------------

def moe_gate_up(x, ids, w1, w1_sf, alpha, wsh, ssh, gssh: float, pairs=None, tokens=None, threads=None):
    """Returns ((act nom, lo, hi), (sact nom, lo, hi), bad_ids).

    act rows are [M*topk, I] (rows for pairs outside ``pairs`` are left 0);
    sact rows are [M, SI] (tokens outside ``tokens`` left 0)."""
    lib = _load()
    x = np.ascontiguousarray(x, np.uint16)
    ids = np.ascontiguousarray(ids, np.int32)
    w1 = np.ascontiguousarray(w1, np.uint8)
    w1_sf = np.ascontiguousarray(w1_sf, np.uint8).reshape(-1)
    alpha = np.ascontiguousarray(alpha, np.float32)
    wsh = np.ascontiguousarray(wsh, np.uint8)
    ssh = np.ascontiguousarray(ssh, np.uint8).reshape(-1)
    M, H = x.shape
    topk = ids.shape[1]
    E, I = w1.shape[0], w1.shape[1] // 2
    SI = wsh.shape[0] // 2
    P = M * topk
    act = [np.zeros((P, I), np.uint16) for _ in range(3)]
    sact = [np.zeros((M, SI), np.uint16) for _ in range(3)]
    t = _threads(threads)
    plist = list(range(P)) if pairs is None else [int(p) for p in pairs]
    tlist = list(range(M)) if tokens is None else [int(v) for v in tokens]
    bad = [0]

    def routed(p):
        tg, tu = np.empty(H, np.float64), np.empty(H, np.float64)
        r = lib.orc_moe_gate_up_routed(_p(x), _p(ids), topk, _p(w1), _p(w1_sf), _p(alpha), E, H, I, p, p + 1,
                                       _p(tg), _p(tu), _p(act[0]), _p(act[1]), _p(act[2]))
        if r:
            bad[0] = 1

    def shared(tok):
        tg, tu = np.empty(H, np.float64), np.empty(H, np.float64)
        lib.orc_moe_gate_up_shared(_p(x), tok, tok + 1, _p(wsh), _p(ssh), float(gssh), H, SI, _p(tg), _p(tu),
                                   _p(sact[0]), _p(sact[1]), _p(sact[2]))

    jobs = [(routed, p) for p in plist] + [(shared, tok) for tok in tlist]
    if t == 1:
        for f, a in jobs:
            f(a)
    else:
        with ThreadPoolExecutor(t) as ex:
            list(ex.map(lambda j: j[0](j[1]), jobs))
    return tuple(act), tuple(sact), bad[0]


def moe_down_combine(act, ids, tw, w2, w2_sf, alpha2, sact, wsd, ssd, gssd: float, tokens=None, threads=None):
    """Returns ((out nom, lo, hi), bad_ids); out is [M, H], rows for tokens
    outside ``tokens`` left 0."""
    lib = _load()
    act = np.ascontiguousarray(act, np.uint16)
    ids = np.ascontiguousarray(ids, np.int32)
    tw = np.ascontiguousarray(tw, np.float32)
    w2 = np.ascontiguousarray(w2, np.uint8)
    w2_sf = np.ascontiguousarray(w2_sf, np.uint8).reshape(-1)
    alpha2 = np.ascontiguousarray(alpha2, np.float32)
    sact = np.ascontiguousarray(sact, np.uint16)
    wsd = np.ascontiguousarray(wsd, np.uint8)
    ssd = np.ascontiguousarray(ssd, np.uint8).reshape(-1)
    M, topk = ids.shape
    E, H, I = w2.shape[0], w2.shape[1], w2.shape[2] * 2
    SI = wsd.shape[1] * 2
    out = [np.zeros((M, H), np.uint16) for _ in range(3)]
    t = _threads(threads)
    tlist = list(range(M)) if tokens is None else [int(v) for v in tokens]
    bad = [0]

    def work(tok):
        tmp = np.empty(max(I, SI), np.float64)
        r = lib.orc_moe_down_combine(_p(act), _p(ids), _p(tw), topk, _p(w2), _p(w2_sf), _p(alpha2), E, H, I,
                                     _p(sact), _p(wsd), _p(ssd), float(gssd), SI, tok, tok + 1, _p(tmp),
                                     _p(out[0]), _p(out[1]), _p(out[2]))
        if r:
            bad[0] = 1

    if t == 1:
        for tok in tlist:
            work(tok)
    else:
        with ThreadPoolExecutor(t) as ex:
            list(ex.map(work, tlist))
    return tuple(out), bad[0]


# --------------------------------------------------------------------------
# Comparison helper (the acceptance rule)
# --------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def check(gpu_bits: np.ndarray, ref, rel: float = 2.0 ** -7, rms_frac: float = 2.0 ** -10):
    """Acceptance rule, per element: |gpu - [lo, hi]| <= rel * |nominal| +
    rms_frac * rms(nominal), the distance to the interval being 0 inside it.
    For an output without an intermediate rounding lo == hi == nominal, so
    this is exactly |gpu - nominal| <= 2^-7 |nominal| + 2^-10 rms(nominal);
    otherwise [lo, hi] holds only the outputs of the intermediates'
    alternative roundings.  Returns (ok, worst_excess, n_bad, first_bad_index)."""
    nom, lo, hi = (bf16_to_f64(r) for r in ref)
    g = bf16_to_f64(gpu_bits)
    lo_, hi_ = np.minimum(lo, hi), np.maximum(lo, hi)
    finite = np.isfinite(nom)
    rms = float(np.sqrt(np.mean(np.square(nom[finite])))) if finite.any() else 0.0
    dist = np.where(g < lo_, lo_ - g, np.where(g > hi_, g - hi_, 0.0))
    tol = rel * np.abs(nom) + rms_frac * rms
    nan_ok = np.isnan(nom) == np.isnan(g)
    bad = (~nan_ok) | (np.nan_to_num(dist, nan=0.0) > tol)
    excess = np.where(bad, np.nan_to_num(dist - tol, nan=np.inf), 0.0)
    nbad = int(bad.sum())
    first = int(np.argmax(bad.reshape(-1))) if nbad else -1
    return nbad == 0, float(excess.max()) if excess.size else 0.0, nbad, first


# --------------------------------------------------------------------------
# W4A4 (activation quantisation, then the NVFP4 x NVFP4 GEMM)
# --------------------------------------------------------------------------

def e4m3_encode(v: float) -> int:
    """Nearest finite E4M3 code of a float v >= 0 (ties to even, saturating at 448)."""
    return int(_load().orc_e4m3_encode(float(v)))


def e2m1_encode(v: float) -> int:
    """Nearest E2M1 code of a float v (ties to even, saturating at 6; zero as +0)."""
    return int(_load().orc_e2m1_encode(float(v)))


def quantize_act(x: np.ndarray, gsi: float) -> tuple[np.ndarray, np.ndarray]:
    """scaled_fp4_quant(x, input_global_scale_inv) as read in the C oracle
    (per 16-value block: s = (amax / 6) * gsi to E4M3, codes = E2M1 of
    x * (gsi / e4m3(s)), all in float): x bf16 bits [M, K] -> (codes uint8
    [M, K / 2], flat 128x4-swizzled scales of scale_bytes(M, K) bytes)."""
    lib = _load()
    x = np.ascontiguousarray(x, np.uint16)
    M, K = x.shape
    assert K % 16 == 0 and gsi > 0
    q = np.empty((M, K // 2), np.uint8)
    sf = np.empty(scale_bytes(M, K), np.uint8)
    lib.orc_quantize_act(_p(x), K, M, K, float(np.float32(gsi)), _p(q), _p(sf))
    return q, sf


def w4a4_gemm(xq: np.ndarray, xsf: np.ndarray, w: np.ndarray, sf: np.ndarray, alpha: float, rows=None,
              threads: int | None = None):
    """The NVFP4 x NVFP4 GEMM of the W4A4 kernels: out = bf16(fp32(xd @ wd^T) *
    alpha) with xd, wd the exact dequantisations of both NVFP4 tensors.  Every
    product e2m1 * e4m3 has at most 5 significant bits, so xd is exact in bf16
    and the GEMM is the dense NVFP4 GEMV of xd (nominal, lo, hi)."""
    xd = dequantize_rows(xq, xsf, threads=threads)
    return nvfp4_gemv(xd, w, sf, alpha, rows=rows, threads=threads)
