"""Thin ctypes binding of libfp4gemv (the C ABI in include/fp4gemv.h).

Argument marshalling only: every call hands device pointers, sizes and the
current CUDA stream of the tensors' device to the library; all computation
runs in the library's kernels.  There is no fallback: importing this module
raises if ``libfp4gemv.so`` is missing and cannot be built, and every call
raises ``Fp4GemvError`` on a non-OK status.

Names follow the pages (vllm.models.flint.ops.nvfp4_gemv: nvfp4_gemv,
bf16_gemv, dequantize_rows; vllm.models.flint.ops.moe_gemv: gate_up,
down_combine): ``nvfp4_gemv`` / ``bf16_gemv`` / ``dequantize_rows`` allocate
and return their output, the MoE pair writes into caller buffers.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

OK = 0
STATUS_NAMES = {
    0: "FP4GEMV_OK",
    1: "FP4GEMV_ERR_INVALID_ARG",
    2: "FP4GEMV_ERR_UNSUPPORTED_SHAPE",
    3: "FP4GEMV_ERR_MISALIGNED",
    4: "FP4GEMV_ERR_CUDA",
    5: "FP4GEMV_ERR_TIMEOUT",
    6: "FP4GEMV_ERR_BAD_INDEX",
}
MAX_M = 128


class Fp4GemvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if not os.path.exists(path) or _build._stale():
        path = _build.build()
    lib = ctypes.CDLL(path)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    sigs = {
        "fp4gemv_scale_bytes": (sz, [i32, i32]),
        "fp4gemv_nvfp4_gemv": (i32, [vp, i64, vp, vp, vp, vp, i64, i32, i32, i32, i32, i32, vp]),
        "fp4gemv_bf16_gemv": (i32, [vp, i64, vp, vp, i64, i32, i32, i32, i32, i32, vp]),
        "fp4gemv_dequantize_rows": (i32, [vp, vp, vp, i32, i32, vp]),
        "fp4gemv_dequantize_rows_padded": (i32, [vp, vp, i32, vp, i32, i32, vp]),
        "fp4gemv_nvfp4_gemv_padded": (i32, [vp, i64, vp, vp, i32, vp, vp, i64, i32, i32, i32, i32, i32, vp]),
        "fp4gemv_dequant_gemm": (i32, [vp, i64, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, vp]),
        "fp4gemv_moe_gate_up": (i32, [vp, vp, i32, i32, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, i32, vp, i32,
                                      vp]),
        "fp4gemv_moe_down_combine_workspace_bytes": (sz, [i32, i32, i32]),
        "fp4gemv_moe_down_combine": (i32, [vp, vp, vp, i32, i32, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, i32,
                                           vp, vp, sz, i32, vp]),
        "fp4gemv_w4a4_workspace_bytes": (sz, [i32, i32]),
        "fp4gemv_quantize_act": (i32, [vp, i64, vp, vp, vp, vp, i32, i32, vp]),
        "fp4gemv_w4a4_gemm": (i32, [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, vp, sz, i32, vp]),
        "fp4gemv_w4a4_linear": (i32, [vp, i64, vp, vp, vp, vp, vp, i64, i32, i32, i32, vp, vp, vp, sz, i32, vp]),
        "fp4gemv_get_device_error": (i32, [vp]),
        "fp4gemv_status_string": (ctypes.c_char_p, [i32]),
        "fp4gemv_set_wait_limit_ns": (i32, [ctypes.c_uint64]),
        "fp4gemv_debug_skip_stage": (i32, [i32]),
        "fp4gemv_launch_count": (ctypes.c_uint64, []),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
LIB_PATH = _build.LIB
_nvfp4_gemv = _lib.fp4gemv_nvfp4_gemv


def lib() -> ctypes.CDLL:
    return _lib


def _check(status: int, what: str) -> None:
    if status != OK:
        raise Fp4GemvError(status, what)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


try:  # the current stream's raw handle without building a Stream object
    _raw_stream = torch._C._cuda_getCurrentRawStream
except AttributeError:  # pragma: no cover - older torch
    def _raw_stream(index):
        return torch.cuda.current_stream(index).cuda_stream


def _stream(dev: torch.device):
    return ctypes.c_void_p(_raw_stream(dev.index if dev.index is not None else torch.cuda.current_device()))


_U8 = torch.uint8
_BF16 = torch.bfloat16
_FP4_WEIGHT_DTYPES = (torch.uint8, torch.int8)
_SCALE_DTYPES = (torch.uint8, torch.float8_e4m3fn)


def _bytes(t: torch.Tensor) -> torch.Tensor:
    """uint8 view of a contiguous tensor (weights, float8 scales)."""
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


def _rows_bf16(x: torch.Tensor, name: str) -> torch.Tensor:
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D bf16 tensor with unit inner stride")
    return x


def flat_scale_buffer(weight_scale: torch.Tensor) -> torch.Tensor:
    """uint8 flat view (no copy) of the storage behind a block-scale tensor.

    A contiguous tensor is its own flat buffer.  A strided view -- the way
    another library may index the same 128x4-swizzled bytes (for instance as
    [rows / 128, K-blocks / 4, 32, 4, 4]) -- must start at offset 0 of its
    storage; the whole storage is then the flat buffer."""
    if weight_scale.element_size() != 1:
        raise ValueError("block scales are one byte each (uint8 / float8_e4m3fn)")
    t = weight_scale if weight_scale.dtype == torch.uint8 else weight_scale.view(torch.uint8)
    if t.is_contiguous():
        return t.reshape(-1)
    if t.storage_offset() != 0:
        raise ValueError("a strided scale view must start at offset 0 of its storage")
    nbytes = t.untyped_storage().nbytes()
    return t.as_strided((nbytes,), (1,), 0)


def scale_bytes(rows: int, K: int) -> int:
    """Bytes of the flat 128x4-swizzled scale buffer of a [rows, K] weight."""
    return int(_lib.fp4gemv_scale_bytes(rows, K))


def nvfp4_gemv(x: torch.Tensor, weight: torch.Tensor, weight_scale: torch.Tensor, global_scale: torch.Tensor,
               silu_mul: bool = False, pdl: bool = True, out: torch.Tensor | None = None,
               sf_k_blocks: int = 0) -> torch.Tensor:
    """bf16 [M, N] = bf16(fp32(x @ dequant(weight).T) * global_scale); with
    silu_mul the [M, N/2] bf16 silu(gate) * up of the [gate | up] halves.

    ``weight_scale``: the flat 128x4-swizzled buffer, or a strided view of one
    (see ``flat_scale_buffer``); ``sf_k_blocks`` > 0 for a buffer whose
    128-row groups hold that many 16-wide K blocks (padded past
    roundup(K / 16, 4)).  The decode path: only cheap attribute checks here
    (the library validates shapes, alignment and pointers before it launches
    anything)."""
    if x.dtype is not _BF16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D bf16 tensor with unit inner stride")
    M, K = x.shape
    if weight.dtype not in _FP4_WEIGHT_DTYPES or weight.dim() != 2 or not weight.is_contiguous() \
            or weight.shape[1] * 2 != K:
        raise ValueError("weight must be a contiguous uint8 [N, K/2] tensor")
    if weight_scale.dtype not in _SCALE_DTYPES:
        raise ValueError("weight_scale must be a uint8 / float8_e4m3fn tensor")
    if not weight_scale.is_contiguous():
        weight_scale = flat_scale_buffer(weight_scale)
    if global_scale.dtype is not torch.float32 or global_scale.numel() != 1:
        raise ValueError("global_scale must be one float32 value")
    N = weight.shape[0]
    n_out = N // 2 if silu_mul else N
    dev = x.device
    if out is None:
        out = torch.empty(M, n_out, dtype=_BF16, device=dev)
    elif out.dtype is not _BF16 or out.dim() != 2 or out.stride(1) != 1 or out.shape[0] != M or out.shape[1] != n_out:
        raise ValueError(f"out must be a bf16 [{M}, {n_out}] tensor with unit inner stride")
    st = _raw_stream(dev.index)
    if sf_k_blocks:
        status = _lib.fp4gemv_nvfp4_gemv_padded(x.data_ptr(), x.stride(0), weight.data_ptr(), weight_scale.data_ptr(),
                                                int(sf_k_blocks), global_scale.data_ptr(), out.data_ptr(),
                                                out.stride(0), M, N, K, 1 if silu_mul else 0, 1 if pdl else 0, st)
        if status:
            raise Fp4GemvError(status, "fp4gemv_nvfp4_gemv_padded")
        return out
    status = _nvfp4_gemv(x.data_ptr(), x.stride(0), weight.data_ptr(), weight_scale.data_ptr(),
                         global_scale.data_ptr(), out.data_ptr(), out.stride(0), M, N, K, 1 if silu_mul else 0,
                         1 if pdl else 0, st)
    if status:
        raise Fp4GemvError(status, "fp4gemv_nvfp4_gemv")
    return out


def bf16_gemv(x: torch.Tensor, weight: torch.Tensor, silu_mul: bool = False, pdl: bool = True,
              out: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 [M, N] = bf16(fp32(x @ weight.T)) for a row-major bf16 [N, K] weight."""
    x = _rows_bf16(x, "x")
    M, K = x.shape
    if weight.dtype != torch.bfloat16 or not weight.is_contiguous() or weight.shape[1] != K:
        raise ValueError("weight must be a contiguous bf16 [N, K] tensor")
    N = weight.shape[0]
    n_out = N // 2 if silu_mul else N
    if out is None:
        out = torch.empty(M, n_out, dtype=torch.bfloat16, device=x.device)
    _check(_lib.fp4gemv_bf16_gemv(_ptr(x), x.stride(0), _ptr(weight), _ptr(out), out.stride(0), M, N, K,
                                  int(silu_mul), int(pdl), _stream(x.device)), "fp4gemv_bf16_gemv")
    return out


def dequantize_rows(weight: torch.Tensor, weight_scale: torch.Tensor,
                    out: torch.Tensor | None = None, sf_k_blocks: int = 0) -> torch.Tensor:
    """Exact bf16 [rows, K] of e2m1 * e4m3 (global scale not applied);
    ``weight_scale`` and ``sf_k_blocks`` as for ``nvfp4_gemv``."""
    w = _bytes(weight)
    rows, K = w.shape[0], w.shape[1] * 2
    if out is None:
        out = torch.empty(rows, K, dtype=torch.bfloat16, device=w.device)
    sf = flat_scale_buffer(weight_scale)
    _check(_lib.fp4gemv_dequantize_rows_padded(_ptr(w), _ptr(sf), int(sf_k_blocks), _ptr(out), rows, K,
                                               _stream(w.device)), "fp4gemv_dequantize_rows")
    return out


def dequant_gemm(x: torch.Tensor, weight: torch.Tensor, weight_scale: torch.Tensor, global_scale: torch.Tensor,
                 w_bf16: torch.Tensor | None = None, out: torch.Tensor | None = None) -> torch.Tensor:
    """dequantize_rows into ``w_bf16`` then bf16(fp32(x @ w_bf16.T) * global_scale)."""
    x = _rows_bf16(x, "x")
    M, K = x.shape
    w = _bytes(weight)
    N = w.shape[0]
    if w_bf16 is None:
        w_bf16 = torch.empty(N, K, dtype=torch.bfloat16, device=x.device)
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _check(_lib.fp4gemv_dequant_gemm(_ptr(x), x.stride(0), _ptr(w), _ptr(_bytes(weight_scale)),
                                     _ptr(global_scale.reshape(1)), _ptr(w_bf16), _ptr(out), out.stride(0), M, N, K,
                                     1, _stream(x.device)), "fp4gemv_dequant_gemm")
    return out


def quantize_act(x: torch.Tensor, input_global_scale_inv: torch.Tensor, x_fp4: torch.Tensor | None = None,
                 x_sf: torch.Tensor | None = None,
                 x_deq: torch.Tensor | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """scaled_fp4_quant of the W4A4 path: bf16 [M, K] -> (uint8 codes [M, K / 2],
    uint8 flat 128x4 block scales of scale_bytes(M, K) bytes); the arithmetic
    is stated in include/fp4gemv.h.  ``x_deq`` (bf16 [M, K], optional)
    receives the exact dequantised values."""
    x = _rows_bf16(x, "x")
    M, K = x.shape
    if x_fp4 is None:
        x_fp4 = torch.empty(M, K // 2, dtype=_U8, device=x.device)
    if x_sf is None:
        x_sf = torch.empty(scale_bytes(M, K), dtype=_U8, device=x.device)
    if x_deq is not None and (x_deq.dtype != torch.bfloat16 or not x_deq.is_contiguous() or
                              tuple(x_deq.shape) != (M, K)):
        raise ValueError("x_deq must be a contiguous bf16 [M, K] tensor")
    _check(_lib.fp4gemv_quantize_act(_ptr(x), x.stride(0), _ptr(input_global_scale_inv.reshape(1)), _ptr(x_fp4),
                                     _ptr(x_sf), _ptr(x_deq), M, K, _stream(x.device)), "fp4gemv_quantize_act")
    return x_fp4, x_sf


def w4a4_workspace_bytes(M: int, K: int) -> int:
    return int(_lib.fp4gemv_w4a4_workspace_bytes(M, K))


def w4a4_gemm(x_fp4: torch.Tensor, x_sf: torch.Tensor, weight: torch.Tensor, weight_scale: torch.Tensor,
              alpha: torch.Tensor, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
              pdl: bool = True) -> torch.Tensor:
    """The W4A4 GEMM: bf16(fp32(xq @ wq.T) * alpha) of NVFP4 activations and weights."""
    xq = _bytes(x_fp4)
    M, K = xq.shape[0], xq.shape[1] * 2
    w = _bytes(weight)
    N = w.shape[0]
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=xq.device)
    if workspace is None:
        workspace = torch.empty(w4a4_workspace_bytes(M, K), dtype=_U8, device=xq.device)
    _check(_lib.fp4gemv_w4a4_gemm(_ptr(xq), _ptr(_bytes(x_sf)), _ptr(w), _ptr(_bytes(weight_scale)),
                                  _ptr(alpha.reshape(1)), _ptr(out), out.stride(0), M, N, K, _ptr(workspace),
                                  workspace.numel(), int(pdl), _stream(xq.device)), "fp4gemv_w4a4_gemm")
    return out


def w4a4_linear(x: torch.Tensor, input_global_scale_inv: torch.Tensor, weight: torch.Tensor,
                weight_scale: torch.Tensor, alpha: torch.Tensor, out: torch.Tensor | None = None,
                x_fp4: torch.Tensor | None = None, x_sf: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, pdl: bool = True) -> torch.Tensor:
    """quantize_act then w4a4_gemm in one call (the quantiser also writes the
    dequantised activations the GEMM reads)."""
    x = _rows_bf16(x, "x")
    M, K = x.shape
    w = _bytes(weight)
    N = w.shape[0]
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    if x_fp4 is None:
        x_fp4 = torch.empty(M, K // 2, dtype=_U8, device=x.device)
    if x_sf is None:
        x_sf = torch.empty(scale_bytes(M, K), dtype=_U8, device=x.device)
    if workspace is None:
        workspace = torch.empty(w4a4_workspace_bytes(M, K), dtype=_U8, device=x.device)
    _check(_lib.fp4gemv_w4a4_linear(_ptr(x), x.stride(0), _ptr(input_global_scale_inv.reshape(1)), _ptr(w),
                                    _ptr(_bytes(weight_scale)), _ptr(alpha.reshape(1)), _ptr(out), out.stride(0), M,
                                    N, K, _ptr(x_fp4), _ptr(x_sf), _ptr(workspace), workspace.numel(), int(pdl),
                                    _stream(x.device)), "fp4gemv_w4a4_linear")
    return out


def moe_gate_up(x, ids, w1, w1_sf, alpha, act, wsh, ssh, gssh, sact, pdl: bool = True) -> None:
    """act[p] = bf16(silu(g) * u) of the routed experts ([up; gate] 64-row
    groups) and sact[t] = the shared expert's silu_mul output, one launch."""
    x = _rows_bf16(x, "x")
    M, H = x.shape
    topk = ids.shape[1]
    E, I = w1.shape[0], w1.shape[1] // 2
    SI = wsh.shape[0] // 2
    _check(_lib.fp4gemv_moe_gate_up(_ptr(x), _ptr(ids), M, topk, _ptr(_bytes(w1)), _ptr(_bytes(w1_sf)), _ptr(alpha),
                                    E, H, I, _ptr(act), _ptr(_bytes(wsh)), _ptr(_bytes(ssh)), _ptr(gssh.reshape(1)),
                                    SI, _ptr(sact), int(pdl), _stream(x.device)), "fp4gemv_moe_gate_up")


def moe_down_combine_workspace_bytes(M: int, topk: int, H: int) -> int:
    return int(_lib.fp4gemv_moe_down_combine_workspace_bytes(M, topk, H))


_workspaces: dict = {}


def moe_workspace(device: torch.device, nbytes: int, stream: int | None = None) -> torch.Tensor:
    """A cached scratch buffer of at least ``nbytes`` for ``device`` and one
    CUDA stream (the current one when ``stream`` is None).  Calls on the same
    stream run one after another and may share it; calls on different
    streams may overlap on the GPU, so each stream gets its own buffer.  It
    needs no initialisation."""
    index = device.index if device.index is not None else torch.cuda.current_device()
    if stream is None:
        stream = _raw_stream(index)
    key = (device.type, index, int(stream))
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def moe_down_combine(act, ids, tw, w2, w2_sf, alpha2, sact, wsd, ssd, gssd, out, pdl: bool = True,
                     workspace: torch.Tensor | None = None) -> None:
    """out[t] = bf16(bf16(sum_j tw[t,j] * y_j) + y_shared): the GEMV grid,
    then (slab kernel) a small combine kernel on the same stream."""
    M, topk = ids.shape
    E, H, I = w2.shape[0], w2.shape[1], w2.shape[2] * 2
    SI = wsd.shape[1] * 2
    need = moe_down_combine_workspace_bytes(M, topk, H)
    if workspace is None:
        workspace = moe_workspace(act.device, need)  # this stream's own buffer
    _check(_lib.fp4gemv_moe_down_combine(_ptr(act), _ptr(ids), _ptr(tw), M, topk, _ptr(_bytes(w2)),
                                         _ptr(_bytes(w2_sf)), _ptr(alpha2), E, H, I, _ptr(sact), _ptr(_bytes(wsd)),
                                         _ptr(_bytes(ssd)), _ptr(gssd.reshape(1)), SI, _ptr(out), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), int(pdl),
                                         _stream(act.device)), "fp4gemv_moe_down_combine")


def get_device_error(device: torch.device | None = None) -> int:
    """Synchronize the current stream, return and clear the device error word
    (0 = FP4GEMV_OK, 5 = timeout, 6 = bad expert id)."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    return int(_lib.fp4gemv_get_device_error(_stream(dev)))


def set_wait_limit_ns(ns: int) -> None:
    """Wait limit of the kernels' bounded waits on the current device (0: the
    built-in 2 s)."""
    _check(_lib.fp4gemv_set_wait_limit_ns(int(ns)), "fp4gemv_set_wait_limit_ns")


def debug_skip_stage(stage: int) -> None:
    """Test hook: the dense GEMV (1 .. 16 tokens) issues nothing for ring stage
    ``stage`` of every CTA, so its wait runs out (-1: off)."""
    _check(_lib.fp4gemv_debug_skip_stage(int(stage)), "fp4gemv_debug_skip_stage")


def launch_count() -> int:
    """Kernel launches issued by the library in this process."""
    return int(_lib.fp4gemv_launch_count())
