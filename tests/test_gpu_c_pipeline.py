"""Workload-level parity: calibration from seeded batches and the full
compress + low-rank backward at the configured sizes.

The oracle calibrates from the same stored bits in fp64; k and R must match
exactly.  For the backward both sides consume the oracle's projector rounded
to the stored dtype, so the comparison isolates the per-step path."""

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import rel, stored, to_dev, to_np, tol, torch_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


def _run_layer(torch, wl, layer, calib_batches):
    from rank_compressed_backprop_gb300 import api

    li = W.LayerInputs(wl, layer)
    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    L, B, Rx, Ry = wl.L, wl.B, wl.Rx, wl.Ry
    Cx, Cy = li.Cx, li.Cy
    x, gy, w = li.x(), li.g_y(), li.w()
    # ---- calibration (a6 + a7) on the GPU vs the oracle ----
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
    assert rel(to_np(CX), CXr) <= 1e-4
    assert rel(to_np(CG), CGr) <= 1e-4
    out = {}
    for name, Cd, Cr, R in (("P", CX, CXr, Rx), ("Q", CG, CGr, Ry)):
        rows = torch.empty(R, L, dtype=dt, device="cuda")
        res = api.calib_solve(Cd, n, rows, eps=wl.eps, p=wl.p, r_override=R, scale_on=True)
        ref = O.calibrate(Cr, n, eps=wl.eps, p=wl.p, r_override=R, scale_on=True)
        auto = O.calibrate(Cr, n, eps=wl.eps, p=wl.p, scale_on=True)
        assert res.k == ref["k"] == auto["k"], name
        assert res.R == R
        out[name] = (res, ref)
    # ---- per-step path with the oracle's projector ----
    Pr = stored(out["P"][1]["rows"], wl.dtype)
    Qr = stored(out["Q"][1]["rows"], wl.dtype)
    PQ = np.concatenate([Pr, Qr], axis=0)
    ref = O.low_rank_backward(x, gy, w, Pr, Qr)
    xd, gd, wd, PQd = to_dev(x), to_dev(gy), to_dev(w), to_dev(PQ)
    xhat = torch.empty(B, Rx, Cx, dtype=dt, device="cuda")
    Sx = torch.empty(B * Rx, Cy, dtype=dt, device="cuda")
    Sq = torch.empty(B * Ry, Cy, dtype=dt, device="cuda")
    gw = torch.empty(Cy, Cx, dtype=torch.float32, device="cuda")
    gx = torch.empty(B, L, Cx, dtype=dt, device="cuda")
    ws = torch.empty(max(api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, dt), 16), dtype=torch.uint8,
                     device="cuda")
    api.compress_act(xd, PQd[:Rx], xhat)
    api.project_grad(gd, PQd, Sx, Sq, Rx, Ry)
    api.grad_w(Sx, xhat, gw, B)
    api.grad_x(Sq, wd, PQd[Rx:], gx, ws)
    torch.cuda.synchronize()
    # both products again through the one-call entry point (one launch where the
    # single-kernel input gradient applies)
    gw1 = torch.full((Cy, Cx), float("nan"), dtype=torch.float32, device="cuda")
    gx1 = torch.full((B, L, Cx), float("nan"), dtype=dt, device="cuda")
    api.grad_w_x(Sx, xhat, gw1, Sq, wd, PQd[Rx:], gx1, ws, B)
    torch.cuda.synchronize()
    errs = {"x_hat": rel(to_np(xhat), ref["x_hat"]), "g_w": rel(to_np(gw), ref["g_w"]),
            "g_x": rel(to_np(gx), ref["g_x"]), "g_w (one call)": rel(to_np(gw1), ref["g_w"]),
            "g_x (one call)": rel(to_np(gx1), ref["g_x"])}
    for k, v in errs.items():
        assert v <= tol(wl.dtype), (k, errs)
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
    wl = W.workload("vit_mlp_pair_49")
    for layer in (0, 1):
        _run_layer(torch, wl, layer, lambda li: [(li.x(), li.g_y())])


def test_bert_ffn_pair(torch):
    # rank 16: 32-column solver blocks; layer 0 (Cy = 3072) takes the cluster-split
    # single-kernel input gradient, layer 1 (Cy = 768) the short one
    wl = W.workload("bert_ffn_pair")
    for layer in (0, 1):
        _run_layer(torch, wl, layer, lambda li: [(li.calib_x(j, 32), li.calib_g(j, 32))
                                                 for j in range(2)])


def test_long_seq_4096_11008(torch):
    # L = 2048 (multi-launch solver), Cy = 11008 (g_hat_x GEMM + expansion).  The
    # statistic is the step's own 4-sample batch: the workload's 64 calibration samples would
    # cost the float64 oracle about 2 TFLOP.
    wl = W.workload("long_seq_4096_11008")
    _run_layer(torch, wl, 0, lambda li: [(li.x(), li.g_y())])
