"""Helpers shared by the GPU parity tests (host-side marshalling only)."""

from __future__ import annotations

import numpy as np
import pytest

import workloads as W

BF16_TOL = 2e-2   # relative Frobenius error, bf16 inputs with fp32 accumulation
F32_TOL = 1e-5    # relative Frobenius error, fp32


def torch_or_skip():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rank_compressed_backprop_gb300.build import build

    build()
    return torch


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_dev(a: np.ndarray):
    """Stored numpy tensor (uint16 bf16 bits or float32) -> CUDA tensor."""
    import torch

    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def to_np(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16(a) -> np.ndarray:
    return W.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def stored(a, dtype: str) -> np.ndarray:
    return bf16(a) if dtype == "bf16" else np.asarray(a, dtype=np.float32)


def rel(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def orthonormal_rows(g: np.random.Generator, R: int, L: int) -> np.ndarray:
    q, _ = np.linalg.qr(g.standard_normal((L, R)))
    return q.T


def tol(dtype: str) -> float:
    return BF16_TOL if dtype == "bf16" else F32_TOL
