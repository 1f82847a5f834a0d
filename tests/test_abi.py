"""The C ABI without a GPU: the library builds/loads, exports every function
the headers in include/ declare, and rejects bad arguments on the host with
the documented status before touching the device."""
import ctypes
import glob
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def fp4():
    from moe_nvfp4_gemv_gb300 import fp4gemv
    return fp4gemv


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(fp4gemv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("fp4gemv_nvfp4_gemv", "fp4gemv_bf16_gemv", "fp4gemv_dequantize_rows", "fp4gemv_moe_gate_up",
                 "fp4gemv_moe_down_combine", "fp4gemv_scale_bytes", "fp4gemv_get_device_error",
                 "fp4gemv_status_string", "fp4gemv_plan_rf", "fp4gemv_plan_tc"):
        assert want in names


def test_library_exports_every_declared_symbol(fp4):
    lib = ctypes.CDLL(fp4.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(fp4):
    for code, name in fp4.STATUS_NAMES.items():
        assert fp4.lib().fp4gemv_status_string(code).decode() == name


@pytest.mark.parametrize("rows,K", [(256, 512), (6144, 4096), (130, 80), (1, 16), (57344, 8192), (0, 64), (16, 8)])
def test_scale_bytes_matches_oracle(fp4, rows, K):
    want = oracle.scale_bytes(rows, K) if rows >= 1 and K >= 16 else 0
    assert fp4.scale_bytes(rows, K) == want


def test_workspace_bytes(fp4):
    # counters (one u64 per 128-row tile, 16-byte padded) + y [M*topk, H] + y_shared [M, H], bf16
    assert fp4.moe_down_combine_workspace_bytes(1, 8, 4096) == 272 + 2 * 8 * 4096 + 2 * 4096
    assert fp4.moe_down_combine_workspace_bytes(0, 8, 4096) == 0


# The library checks sizes and flags first, then alignment (a null pointer is
# aligned), then null pointers.  So every call below passes NULL for each
# pointer that is not the subject of the test: if a check regressed, the
# null-pointer check still returns FP4GEMV_ERR_INVALID_ARG before anything
# could launch.  Only the null-pointer tests need the other pointers to be
# non-null; they use a fabricated address and run only where no CUDA device
# is visible, so a regression there cannot reach a GPU.
A16 = 1 << 20  # a fabricated, 16-byte aligned "device address"
try:
    import torch
    _GPU_VISIBLE = torch.cuda.is_available()
except Exception:  # pragma: no cover - torch is part of the image
    _GPU_VISIBLE = False
no_gpu_only = pytest.mark.skipif(_GPU_VISIBLE, reason="fabricated device addresses: run only without a GPU")


def gemv(fp4, x=0, ldx=512, w=0, sf=0, gs=0, out=0, ldo=256, M=1, N=256, K=512, silu=0, pdl=1):
    vp = ctypes.c_void_p
    return fp4.lib().fp4gemv_nvfp4_gemv(vp(x), ldx, vp(w), vp(sf), vp(gs), vp(out), ldo, M, N, K, silu, pdl, None)


@pytest.mark.parametrize("kw,status", [
    (dict(M=0), 1), (dict(silu=2), 1), (dict(pdl=3), 1), (dict(ldx=256), 1), (dict(ldo=128), 1),
    (dict(M=129), 2), (dict(N=264), 2), (dict(N=272, ldo=272, silu=1), 2), (dict(K=480, ldx=512), 2),
    (dict(K=128, ldx=128), 2),
    (dict(x=A16 + 2), 3), (dict(ldx=516), 3), (dict(w=A16 + 8), 3), (dict(sf=A16 + 4), 3),
    (dict(out=A16 + 2), 3), (dict(ldo=260), 3), (dict(gs=A16 + 2), 3),
    (dict(), 1),
])
def test_nvfp4_gemv_host_validation(fp4, kw, status):
    assert gemv(fp4, **kw) == status


@no_gpu_only
@pytest.mark.parametrize("null", ["x", "w", "sf", "gs", "out"])
def test_nvfp4_gemv_null_pointers(fp4, null):
    kw = dict(x=A16, w=A16, sf=A16, gs=A16, out=A16)
    kw[null] = 0
    assert gemv(fp4, **kw) == 1


def test_dequantize_rows_host_validation(fp4):
    vp = ctypes.c_void_p
    f = fp4.lib().fp4gemv_dequantize_rows
    assert f(vp(0), vp(0), vp(0), 16, 256, None) == 1
    assert f(vp(0), vp(0), vp(0), 8, 256, None) == 2   # rows % 16
    assert f(vp(0), vp(0), vp(0), 16, 320, None) == 2  # K % 256
    assert f(vp(A16 + 1), vp(0), vp(0), 16, 256, None) == 3


def test_moe_host_validation(fp4):
    vp = ctypes.c_void_p
    L = fp4.lib()
    a = [vp(0)] * 16
    # gate_up: M*topk > 1024, then H % 64, then a null pointer
    assert L.fp4gemv_moe_gate_up(a[0], a[1], 200, 8, a[2], a[3], a[4], 128, 4096, 1536, a[5], a[6], a[7], a[8], 1536,
                                 a[9], 1, None) == 2
    assert L.fp4gemv_moe_gate_up(a[0], a[1], 1, 8, a[2], a[3], a[4], 128, 4100, 1536, a[5], a[6], a[7], a[8], 1536,
                                 a[9], 1, None) == 2
    assert L.fp4gemv_moe_gate_up(a[0], a[1], 1, 8, a[2], a[3], a[4], 128, 4096, 1536, a[5], a[6], a[7], a[8], 1536,
                                 a[9], 1, None) == 1
    assert L.fp4gemv_moe_gate_up(vp(A16 + 4), a[1], 1, 8, a[2], a[3], a[4], 128, 4096, 1536, a[5], a[6], a[7], a[8],
                                 1536, a[9], 1, None) == 3
    # down_combine: workspace too small, then a null pointer
    assert L.fp4gemv_moe_down_combine(a[0], a[1], a[2], 1, 8, a[3], a[4], a[5], 128, 4096, 1536, a[6], a[7], a[8],
                                      a[9], 1536, a[10], a[11], 16, 1, None) == 1
    assert L.fp4gemv_moe_down_combine(a[0], a[1], a[2], 1, 8, a[3], a[4], a[5], 128, 4096, 1536, a[6], a[7], a[8],
                                      a[9], 100, a[10], a[11], 1 << 24, 1, None) == 2
    assert L.fp4gemv_moe_down_combine(a[0], a[1], a[2], 1, 8, a[3], a[4], a[5], 128, 4096, 1536, a[6], a[7], a[8],
                                      a[9], 1536, a[10], a[11], 1 << 24, 1, None) == 1


def test_w4a4_host_validation(fp4):
    vp = ctypes.c_void_p
    L = fp4.lib()
    z = vp(0)
    assert fp4.w4a4_workspace_bytes(3, 512) == 3 * 512 * 2 and fp4.w4a4_workspace_bytes(0, 512) == 0
    # quantize_act: ldx < K, then K % 16, then misaligned x, then a null pointer
    assert L.fp4gemv_quantize_act(z, 8, z, z, z, z, 1, 16, None) == 1
    assert L.fp4gemv_quantize_act(z, 24, z, z, z, z, 1, 24, None) == 2
    assert L.fp4gemv_quantize_act(vp(A16 + 2), 16, z, z, z, z, 1, 16, None) == 3
    assert L.fp4gemv_quantize_act(z, 16, z, z, z, z, 1, 16, None) == 1
    # w4a4_gemm: K < 256, then the workspace too small, then a null pointer
    assert L.fp4gemv_w4a4_gemm(z, z, z, z, z, z, 16, 1, 16, 128, z, 1 << 20, 1, None) == 2
    assert L.fp4gemv_w4a4_gemm(z, z, z, z, z, z, 16, 4, 16, 256, z, 1024, 1, None) == 1
    assert L.fp4gemv_w4a4_gemm(z, z, z, z, z, z, 16, 4, 16, 256, z, 1 << 20, 1, None) == 1
    assert L.fp4gemv_w4a4_linear(z, 256, z, z, z, z, z, 16, 4, 16, 256, z, z, z, 1 << 20, 2, None) == 1


def test_launch_counter_starts_at_zero_without_launches(fp4):
    assert fp4.launch_count() >= 0
