"""Edge cases of the per-step path and of the calibration: full-rank
projectors (the method reduces to exact backpropagation), a single token,
the largest ranks, and rank-deficient statistics."""

import numpy as np
import pytest

import oracle as O
from gpu_util import (assert_parity, nan_like, orthonormal_rows, rel, rng, stored, to_dev, to_np,
                      tol, torch_or_skip)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


def _tdt(torch, dtype):
    return torch.float32 if dtype == "f32" else torch.bfloat16


def _step(torch, dtype, x, gy, w, P, Q):
    """compress + project + both gradients through the library."""
    from rank_compressed_backprop_gb300 import api

    B, L, Cx = x.shape
    Cy = w.shape[0]
    Rx, Ry = P.shape[0], Q.shape[0]
    dt = _tdt(torch, dtype)
    PQ = np.concatenate([P, Q], axis=0)
    xd, gd, wd, PQd = to_dev(x), to_dev(gy), to_dev(w), to_dev(PQ)
    xhat = nan_like(torch, (B, Rx, Cx), dt)
    Sx = nan_like(torch, (B * Rx, Cy), dt)
    Sq = nan_like(torch, (B * Ry, Cy), dt)
    gw = nan_like(torch, (Cy, Cx), torch.float32)
    gx = nan_like(torch, (B, L, Cx), dt)
    ws = torch.empty(max(api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, dt), 16), dtype=torch.uint8,
                     device="cuda")
    api.compress_act(xd, PQd[:Rx], xhat)
    api.project_grad(gd, PQd, Sx, Sq, Rx, Ry)
    api.grad_w_x(Sx, xhat, gw, Sq, wd, to_dev(Q), gx, ws, B)
    torch.cuda.synchronize()
    return to_np(xhat), to_np(gw), to_np(gx)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_full_rank_projectors_reproduce_vanilla_backprop(torch, dtype):
    # R = L with orthonormal P and Q: P^T P = Q^T Q = I, so g_w = sum_b g_y,b^T x_b
    # and g_tilde_x = g_y w exactly (up to the storage rounding of P and Q)
    g = rng(2100)
    B, L, Cx, Cy = 3, 32, 64, 72
    x = stored(g.standard_normal((B, L, Cx)), dtype)
    gy = stored(g.standard_normal((B, L, Cy)), dtype)
    w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), dtype)
    P = stored(orthonormal_rows(g, L, L), dtype)
    Q = stored(orthonormal_rows(g, L, L), dtype)
    _, gw, gx = _step(torch, dtype, x, gy, w, P, Q)
    ref = O.vanilla_backward(x, gy, w)
    bound = 1e-5 if dtype == "f32" else 3e-2   # bf16 projectors are orthonormal to ~4e-3
    assert_parity(gw, ref["g_w"], bound, "g_w")
    assert_parity(gx, ref["g_x"], bound, "g_x")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,L,Cx,Cy,R", [(2, 1, 64, 64, 1),      # a single token
                                        (2, 130, 64, 136, 64),  # the largest ranks
                                        (1, 64, 8, 8, 4)])      # the narrowest bf16 rows
def test_edge_shapes_match_the_oracle(torch, dtype, B, L, Cx, Cy, R):
    g = rng(2200 + L + R)
    x = stored(g.standard_normal((B, L, Cx)), dtype)
    gy = stored(g.standard_normal((B, L, Cy)), dtype)
    w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), dtype)
    P = stored(orthonormal_rows(g, R, L), dtype)
    Q = stored(orthonormal_rows(g, R, L), dtype)
    xh, gw, gx = _step(torch, dtype, x, gy, w, P, Q)
    ref = O.low_rank_backward(x, gy, w, P, Q)
    for name, got, want in (("x_hat", xh, ref["x_hat"]), ("g_w", gw, ref["g_w"]),
                            ("g_x", gx, ref["g_x"])):
        assert_parity(got, want, tol(dtype), name)


@pytest.mark.parametrize("L,multi", [(48, False),     # full Jacobi
                                     (200, False),    # one-launch cluster, basis gathered
                                     (700, False),    # one-launch cluster, basis through L2
                                     (700, True)])    # multi-launch loop
def test_rank_one_statistic(torch, monkeypatch, L, multi):
    """C = n v v^T: one non-zero eigenvalue, so k = 1 and the other R - 1 rows
    span zero eigenvalues (their block is rank-deficient for the Cholesky-QR,
    which must fall back to the Jacobi form)."""
    from rank_compressed_backprop_gb300 import api

    if multi:
        monkeypatch.setenv("INSTANT_SOLVER_MULTI", "1")
    g = rng(2300 + L)
    v = g.standard_normal(L)
    v /= np.linalg.norm(v)
    n = 16
    C = (n * 3.0 * np.outer(v, v)).astype(np.float32)
    rows = torch.full((4, L), 9.0, dtype=torch.float32, device="cuda")
    res = api.calib_solve(to_dev(C), n, rows, eps=0.95, p=2, r_override=0, scale_on=True)
    assert (res.k, res.R) == (1, 3)
    assert abs(res.eigenvalues[0] - 3.0) <= 1e-4 * 3.0
    assert abs(res.energy - 9.0) <= 1e-6 * 9.0
    got = to_np(rows)
    assert np.isfinite(got).all()
    # row 0 = s * v with the sign that makes the largest entry positive, s = 1/3
    v = v if v[np.argmax(np.abs(v))] > 0 else -v
    assert np.max(np.abs(got[0] - v / 3.0)) <= 1e-4
    # rows 1 and 2 complete an orthonormal set (scaled by s) in the null space
    assert np.max(np.abs(got[:3] @ got[:3].T - np.eye(3) / 9.0)) <= 1e-4
    assert np.max(np.abs(got[1:3] @ v)) <= 1e-4
    assert np.all(got[3] == 0)
    assert api.device_status() == 0
