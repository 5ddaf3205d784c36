"""Workload-level parity: calibration from seeded batches and the full
compress + low-rank backward at the configured sizes.

The oracle calibrates from the same stored bits in fp64; k and R must match
exactly, and where the spectrum separates the kept eigenvectors from the rest
the GPU's projector rows must match the oracle's.  For the backward both sides
consume the oracle's projector rounded to the stored dtype, so the comparison
isolates the per-step path.  Every output starts as NaN and is compared
element by element (finite, relative Frobenius, per row, largest element)."""

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import assert_parity, nan_like, stored, to_dev, to_np, tol, torch_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


def k_margin(ref, eps):
    """Distance of the energy rule's decision from its threshold, relative to
    E: how far the cumulative energy at k lies above eps*E, and at k-1 below."""
    lam, E, k = ref["eigenvalues"], ref["energy"], ref["k"]
    cum = np.cumsum(np.asarray(lam, np.float64) ** 2)
    above = (cum[k - 1] - eps * E) / E
    below = (eps * E - cum[k - 2]) / E if k >= 2 else np.inf
    return float(min(above, below))


def _calibrate(torch, wl, li, calib_batches, compare_rows):
    """Accumulates both statistics batch by batch on the GPU and in the oracle,
    solves them on both sides and checks k, R (exact), the statistics and,
    if asked, the projector rows."""
    from rank_compressed_backprop_gb300 import api

    L, Rx, Ry = wl.L, wl.Rx, wl.Ry
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    CX = torch.zeros(L, L, dtype=torch.float32, device="cuda")
    CG = torch.zeros(L, L, dtype=torch.float32, device="cuda")
    CXr = np.zeros((L, L))
    CGr = np.zeros((L, L))
    n = 0
    for xc, gc in calib_batches(li):
        api.calib_accumulate(to_dev(xc), CX)
        api.calib_accumulate(to_dev(gc), CG)
        CXr = O.accumulate_autocorrelation(xc, CXr)
        CGr = O.accumulate_autocorrelation(gc, CGr)
        n += xc.shape[0]
    assert_parity(to_np(CX), CXr, 1e-4, "C_X")
    assert_parity(to_np(CG), CGr, 1e-4, "C_G")
    out = {}
    for name, Cd, Cr, R in (("P", CX, CXr, Rx), ("Q", CG, CGr, Ry)):
        rows = nan_like(torch, (R, L), dt)
        res = api.calib_solve(Cd, n, rows, eps=wl.eps, p=wl.p, r_override=R, scale_on=True)
        ref = O.calibrate(Cr, n, eps=wl.eps, p=wl.p, r_override=R, scale_on=True)
        auto = O.calibrate(Cr, n, eps=wl.eps, p=wl.p, scale_on=True)
        m = k_margin(ref, wl.eps)
        print(f"{wl.name} {name}: n={n} k={res.k} (oracle {ref['k']}), R_auto={auto['R']}, "
              f"k margin {m:.3e} of E")
        assert res.k == ref["k"] == auto["k"], name
        assert res.R == R
        assert abs(res.scale - ref["scale"]) <= 1e-4 * ref["scale"], name
        got = to_np(rows)
        assert np.isfinite(got).all(), name
        if compare_rows:
            # s * u_i^T with canonical signs, compared scale-free
            lim = 2e-3 if wl.dtype == "f32" else 1.5e-2
            err = np.max(np.abs(got / ref["scale"] - ref["rows"] / ref["scale"]))
            assert err <= lim, (name, err)
        out[name] = (res, ref, auto, m)
    return out, n


def _run_layer(torch, wl, layer, calib_batches, compare_rows=True):
    from rank_compressed_backprop_gb300 import api

    li = W.LayerInputs(wl, layer)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    L, B, Rx, Ry = wl.L, wl.B, wl.Rx, wl.Ry
    Cx, Cy = li.Cx, li.Cy
    # ---- calibration (a6 + a7) on the GPU vs the oracle ----
    out, _ = _calibrate(torch, wl, li, calib_batches, compare_rows)
    # ---- per-step path with the oracle's projector ----
    x, gy, w = li.x(), li.g_y(), li.w()
    Pr = stored(out["P"][1]["rows"], wl.dtype)
    Qr = stored(out["Q"][1]["rows"], wl.dtype)
    PQ = np.concatenate([Pr, Qr], axis=0)
    ref = O.low_rank_backward(x, gy, w, Pr, Qr)
    xd, gd, wd, PQd = to_dev(x), to_dev(gy), to_dev(w), to_dev(PQ)
    xhat = nan_like(torch, (B, Rx, Cx), dt)
    Sx = nan_like(torch, (B * Rx, Cy), dt)
    Sq = nan_like(torch, (B * Ry, Cy), dt)
    gw = nan_like(torch, (Cy, Cx), torch.float32)
    gx = nan_like(torch, (B, L, Cx), dt)
    ws = torch.full((max(api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, dt), 16),), 255,
                    dtype=torch.uint8, device="cuda")
    api.compress_act(xd, PQd[:Rx], xhat)
    api.project_grad(gd, PQd, Sx, Sq, Rx, Ry)
    api.grad_w(Sx, xhat, gw, B)
    api.grad_x(Sq, wd, PQd[Rx:], gx, ws)
    torch.cuda.synchronize()
    # both products again through the one-call entry point (one launch where the
    # single-kernel input gradient applies)
    gw1 = nan_like(torch, (Cy, Cx), torch.float32)
    gx1 = nan_like(torch, (B, L, Cx), dt)
    api.grad_w_x(Sx, xhat, gw1, Sq, wd, PQd[Rx:], gx1, ws, B)
    torch.cuda.synchronize()
    t = tol(wl.dtype)
    errs = {
        "x_hat": assert_parity(to_np(xhat), ref["x_hat"], t, "x_hat"),
        "Sx": assert_parity(to_np(Sx).reshape(B, Rx, Cy), ref["Sx"], t, "Sx"),
        "Sq": assert_parity(to_np(Sq).reshape(B, Ry, Cy), ref["Sq"], t, "Sq"),
        "g_w": assert_parity(to_np(gw), ref["g_w"], t, "g_w"),
        "g_x": assert_parity(to_np(gx), ref["g_x"], t, "g_x"),
        "g_w (one call)": assert_parity(to_np(gw1), ref["g_w"], t, "g_w (one call)"),
        "g_x (one call)": assert_parity(to_np(gx1), ref["g_x"], t, "g_x (one call)"),
    }
    assert api.device_status() == 0
    return out, errs


def test_fp32_linear_64(torch):
    wl = W.workload("fp32_linear_64")
    out, errs = _run_layer(torch, wl, 0, lambda li: [(li.calib_x(0, 8), li.calib_g(0, 8))])
    # planted 2^-i spectrum: k = 2 and k + p = 4 = the workload's rank
    assert out["P"][0].k == 2 and out["Q"][0].k == 2


def test_bert_base_block(torch):
    wl = W.workload("bert_base_block")
    _run_layer(torch, wl, 0, lambda li: [(li.calib_x(j, 32), li.calib_g(j, 32)) for j in range(2)])


def test_vit_mlp_pair_49(torch):
    # GELU activations: eigenvalues 2..49 of C_X lie within ~1e-3 of each other and
    # the g_y statistic keeps noise modes beyond its planted rank 6, so the rows are
    # not unique; k, the eigenvalues and the backward given the oracle's rows are
    wl = W.workload("vit_mlp_pair_49")
    for layer in (0, 1):
        _run_layer(torch, wl, layer, lambda li: [(li.x(), li.g_y())], compare_rows=False)


def test_bert_ffn_pair(torch):
    # rank 16: 32-column solver blocks; layer 0 (Cy = 3072) takes the cluster-split
    # single-kernel input gradient, layer 1 (Cy = 768) the short one
    wl = W.workload("bert_ffn_pair")
    for layer in (0, 1):
        _run_layer(torch, wl, layer, lambda li: [(li.calib_x(j, 32), li.calib_g(j, 32))
                                                 for j in range(2)])


def test_long_seq_4096_11008(torch):
    # L = 2048 (multi-launch solver), Cy = 11008 (g_hat_x GEMM + expansion); the
    # statistic here is the step's own 4-sample batch (the configured 64-sample
    # statistic has a test of its own below)
    wl = W.workload("long_seq_4096_11008")
    _run_layer(torch, wl, 0, lambda li: [(li.x(), li.g_y())])


def test_long_seq_4096_11008_calibration_64_samples(torch):
    """The long-sequence layer's calibration at its configured statistic: 64
    samples of x [2048, 4096] and g_y [2048, 11008] accumulated in 16 chunks of 4
    on both sides (about 8 TFLOP of float64 products in the oracle), then the
    energy rule at eps = 0.95, p = 4: k and R_auto = k + p exact, and the top-16
    rows of both projectors within the bf16 row tolerance."""
    wl = W.workload("long_seq_4096_11008")
    assert wl.calib_samples == 64 and wl.p == 4
    chunks = wl.calib_samples // 4
    out, n = _calibrate(torch, wl, W.LayerInputs(wl, 0),
                        lambda li: ((li.calib_x(j, 4), li.calib_g(j, 4)) for j in range(chunks)),
                        compare_rows=True)
    assert n == 64
    for name in ("P", "Q"):
        res, ref, auto, m = out[name]
        assert auto["R"] == min(res.k + wl.p, wl.L)
        assert m > 0
