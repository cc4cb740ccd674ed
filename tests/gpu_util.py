"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

import workloads

# GEMM tolerance for bf16 inputs with fp32 accumulation, elementwise:
# |gpu - oracle| <= ATOL + RTOL * |oracle|.
ATOL = 2e-2
RTOL = 1e-2


def bits(t: torch.Tensor) -> np.ndarray:
    return workloads.bf16_bits(t)


def as_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def assert_close(gpu_bf16: torch.Tensor, oracle_f32: np.ndarray, what: str = ""):
    g = as_f32(gpu_bf16)
    o = np.asarray(oracle_f32, dtype=np.float32)
    assert g.shape == o.shape, (g.shape, o.shape)
    err = np.abs(g.astype(np.float64) - o)
    bound = ATOL + RTOL * np.abs(o)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; first at {tuple(i)}: "
                             f"gpu {g[tuple(i)]} oracle {o[tuple(i)]}; max abs err {err.max():.4g}")


def rel_frobenius(gpu_bf16: torch.Tensor, oracle_f32: np.ndarray) -> float:
    g = as_f32(gpu_bf16).astype(np.float64)
    o = np.asarray(oracle_f32, dtype=np.float64)
    return float(np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-30))
