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


def nan_like(torch, shape, dtype):
    """An output buffer filled with NaN, so that an element the kernel never
    writes fails the finiteness check."""
    return torch.full(tuple(shape), float("nan"), dtype=dtype, device="cuda")


def parity_errors(got, ref) -> dict:
    """Element-level error figures of ``got`` against ``ref`` (rows = last axis)."""
    a = np.asarray(got, np.float64)
    b = np.asarray(ref, np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    d = (a - b).reshape(-1, a.shape[-1]) if a.ndim else (a - b).reshape(1, 1)
    rb = b.reshape(d.shape)
    row_err = np.sqrt(np.sum(d * d, axis=1))
    row_ref = np.sqrt(np.sum(rb * rb, axis=1))
    rms_row = float(np.sqrt(np.mean(row_ref * row_ref))) if row_ref.size else 0.0
    nb = float(np.linalg.norm(b))
    worst = int(np.argmax(row_err / (row_ref + rms_row + 1e-300))) if row_err.size else 0
    return {
        "finite": bool(np.isfinite(a).all()),
        "rel": float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)),
        "max_abs": float(np.max(np.abs(a - b))) if a.size else 0.0,
        "max_ref": float(np.max(np.abs(b))) if b.size else 0.0,
        "row_ratio": float(row_err[worst] / (row_ref[worst] + rms_row)) if row_err.size and rms_row > 0
        else float(row_err.max() if row_err.size else 0.0),
        "worst_row": worst,
    }


def assert_parity(got, ref, tolerance: float, what: str = "") -> dict:
    """Parity of one output against the oracle, element by element.

    * every element finite (outputs start as NaN, so an unwritten one fails);
    * relative Frobenius error ``<= tolerance``;
    * every row (last axis: one token, rank or channel row of one sample)
      within ``2 * tolerance * (||ref_row|| + rms row norm)``: a single wrong row
      cannot hide in the norm of a large batch;
    * the largest element error ``<= 8 * tolerance * max |ref|``."""
    e = parity_errors(got, ref)
    assert e["finite"], (what, "non-finite (unwritten?) elements", e)
    assert e["rel"] <= tolerance, (what, e)
    assert e["row_ratio"] <= 2 * tolerance, (what, e)
    assert e["max_abs"] <= 8 * tolerance * e["max_ref"] + 1e-300, (what, e)
    return e
