"""Reconstruction error of the gradient compression while its subspace drifts.

Between two recalibrations (every ``N_t`` steps, page "INSTANT: Compressing
Gradients and Activations for Resource-Efficient Training", 整体框架) the
projector Q stays fixed while the output gradients move; the oversampling p
of 关键设计 2 (R = k + p rows instead of k) is what keeps Q useful meanwhile.
This module measures that: per step, ``||g_y - Q^T Q g_y|| / ||g_y||`` with the
projector solved without scaling (orthonormal rows).

Every computation runs in the CUDA library (calib_accumulate, calib_solve,
compress_act and reconstruction_error); torch only owns the buffers.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Callable

import torch

from . import api


@dataclasses.dataclass
class DriftRun:
    p: int
    n_t: int
    errors: list            # per step: ||g - Q^T Q g|| / ||g||
    calibrations: list      # (step, k, R) of every recalibration


def drift_errors(batch: Callable[[int], torch.Tensor], steps: int, n_t: int, p: int, *,
                 eps: float = 0.95, r_cap: int = 16) -> DriftRun:
    """Runs ``steps`` steps on the batches ``batch(step)`` (device tensors
    ``[B, L, C]``, bf16 or fp32), recalibrating Q from the step's own batch every
    ``n_t`` steps with oversampling ``p``; returns the per-step errors."""
    if steps < 1 or n_t < 1 or p < 0:
        raise ValueError("drift_errors: steps, n_t >= 1 and p >= 0")
    g = batch(0)
    B, L, C = g.shape
    dev, dt = g.device, g.dtype
    r_cap = min(r_cap, L)
    C_sum = torch.zeros(L, L, dtype=torch.float32, device=dev)
    Q = torch.zeros(r_cap, L, dtype=dt, device=dev)
    S = torch.empty(B * r_cap * C, dtype=dt, device=dev)
    ws = torch.empty(api.calib_workspace_bytes(L, r_cap), dtype=torch.uint8, device=dev)
    ws_err = torch.empty(16, dtype=torch.uint8, device=dev)
    errors, cals = [], []
    R = 0
    for t in range(steps):
        if t:
            g = batch(t)
        if t % n_t == 0:
            C_sum.zero_()
            api.calib_accumulate(g, C_sum)
            res = api.calib_solve(C_sum, B, Q, eps=eps, p=p, r_override=0, scale_on=False, ws=ws)
            R = res.R
            cals.append((t, res.k, res.R))
        Qr = Q[:R]
        Sr = S[: B * R * C]
        api.compress_act(g, Qr, Sr.view(B, R, C))
        e2, n2 = api.reconstruction_error(g, Qr, Sr.view(B * R, C), ws_err)
        errors.append(math.sqrt(e2 / n2) if n2 > 0 else 0.0)
    return DriftRun(p, n_t, errors, cals)
