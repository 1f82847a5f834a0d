"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import pytest
import torch

import oracle
from moe_nvfp4_gemv_gb300 import synth


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def dense_inputs(M, N, K, seed=0):
    """(x bf16 [M,K], w u8 [N,K/2], sf u8 flat) on the CPU."""
    w = synth.fp4_bytes(N, K, seed=seed + 1)
    sf = synth.e4m3_bytes(oracle.scale_bytes(N, K), seed=seed + 2)
    x = synth.activations(M, K, seed=seed + 3)
    return x, w, sf


def assert_close(gpu_bits, ref, what=""):
    ok, excess, nbad, first = oracle.check(gpu_bits, ref)
    if not ok:
        nom = oracle.bf16_to_f64(ref[0]).reshape(-1)
        g = oracle.bf16_to_f64(gpu_bits).reshape(-1)
        raise AssertionError(f"{what}: {nbad} of {g.size} outside tolerance (worst excess {excess:.3g}); "
                             f"first at {first}: gpu {g[first]!r} ref {nom[first]!r}")


def sample_rows(n, count, seed):
    rng = np.random.default_rng(seed)
    rows = set([0, n - 1, n // 2]) | set(rng.integers(0, n, size=count).tolist())
    return np.array(sorted(rows), np.int64)
