"""Per-entry-point parity of the CUDA library against the fp64 oracle.

Shapes span several tiles and a ragged tail in every tiled dimension.  The
fp32 cases (plain FFMA kernels) run first, then the bf16 tcgen05 kernels.
"""

import numpy as np
import pytest

import oracle as O
from gpu_util import (assert_parity, nan_like, orthonormal_rows, rel, rng, stored, to_dev, to_np,
                      tol, torch_or_skip)

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "bf16"]


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


def _api():
    from rank_compressed_backprop_gb300 import api

    return api


def _tdt(torch, dtype):
    return torch.float32 if dtype == "f32" else torch.bfloat16


# --------------------------------------------------------------------------
# compress_act / project_grad
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("B,L,C,Rx", [(1, 64, 64, 4), (3, 200, 392, 8), (2, 49, 448, 8),
                                      (2, 130, 264, 16), (1, 512, 136, 5)])
def test_compress_act(torch, dtype, B, L, C, Rx):
    g = rng(100 + L + C)
    x = stored(g.standard_normal((B, L, C)), dtype)
    P = stored(orthonormal_rows(g, Rx, L), dtype)
    xh = nan_like(torch, (B, Rx, C), _tdt(torch, dtype))
    _api().compress_act(to_dev(x), to_dev(P), xh)
    torch.cuda.synchronize()
    ref = O.compress_act(x, P)
    assert_parity(to_np(xh), ref, tol(dtype), "x_hat")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("B,L,C,Rx,Ry", [(1, 64, 64, 4, 4), (3, 200, 392, 5, 7),
                                         (2, 49, 448, 8, 8), (2, 300, 256, 16, 16),
                                         (1, 2048, 264, 16, 16), (2, 96, 128, 24, 40)])
def test_project_grad(torch, dtype, B, L, C, Rx, Ry):
    g = rng(200 + L + C + Rx)
    gy = stored(g.standard_normal((B, L, C)), dtype)
    PQ = stored(orthonormal_rows(g, Rx + Ry, L), dtype)
    dt = _tdt(torch, dtype)
    Sx = nan_like(torch, (B * Rx, C), dt)
    Sq = nan_like(torch, (B * Ry, C), dt)
    _api().project_grad(to_dev(gy), to_dev(PQ), Sx, Sq, Rx, Ry)
    torch.cuda.synchronize()
    rx, rq = O.project_grad(gy, PQ[:Rx], PQ[Rx:])
    assert_parity(to_np(Sx).reshape(B, Rx, C), rx, tol(dtype), "Sx")
    assert_parity(to_np(Sq).reshape(B, Ry, C), rq, tol(dtype), "Sq")


# --------------------------------------------------------------------------
# grad_w
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("B,Rx,Cx,Cy", [(1, 4, 64, 64), (5, 8, 200, 328), (32, 8, 768, 768),
                                        (3, 16, 520, 136), (1, 3, 72, 48)])
@pytest.mark.parametrize("accumulate", [False, True])
def test_grad_w(torch, dtype, B, Rx, Cx, Cy, accumulate):
    g = rng(300 + B + Cx + Cy)
    Sx = stored(g.standard_normal((B * Rx, Cy)), dtype)
    xh = stored(g.standard_normal((B, Rx, Cx)), dtype)
    gw0 = g.standard_normal((Cy, Cx)).astype(np.float32)
    gw = to_dev(gw0) if accumulate else nan_like(torch, (Cy, Cx), torch.float32)
    _api().grad_w(to_dev(Sx), to_dev(xh), gw, B, accumulate=accumulate)
    torch.cuda.synchronize()
    ref = O.grad_w(O.decode(Sx).reshape(B, Rx, Cy), O.decode(xh))
    if accumulate:
        ref = ref + gw0.astype(np.float64)
    assert_parity(to_np(gw), ref, 1e-5 if dtype == "f32" else 2e-3, "g_w")


# --------------------------------------------------------------------------
# grad_x (g_hat_x = Sq w, then the rank-R expansion)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("B,L,Cx,Cy,Ry", [(1, 64, 64, 64, 4), (3, 150, 272, 520, 8),
                                          (2, 49, 448, 1792, 8), (2, 300, 1024, 256, 16),
                                          (1, 200, 136, 72, 32), (4, 130, 2056, 64, 16)])
def test_grad_x(torch, dtype, B, L, Cx, Cy, Ry):
    api = _api()
    g = rng(400 + L + Cx + Cy)
    Sq = stored(g.standard_normal((B * Ry, Cy)), dtype)
    w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), dtype)
    Q = stored(orthonormal_rows(g, Ry, L), dtype)
    dt = _tdt(torch, dtype)
    gx = nan_like(torch, (B, L, Cx), dt)
    ws = torch.empty(max(api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, dt), 16), dtype=torch.uint8,
                     device="cuda")
    api.grad_x(to_dev(Sq), to_dev(w), to_dev(Q), gx, ws)
    torch.cuda.synchronize()
    ref = O.grad_x(O.decode(Sq).reshape(B, Ry, Cy), w, Q)
    assert_parity(to_np(gx), ref, tol(dtype), "g_x")


# --------------------------------------------------------------------------
# calib_accumulate
# --------------------------------------------------------------------------
def _syrk_tiles(monkeypatch, tiles):
    """128 x 256 tiles (forced for any L > 128) or 128 x 128 (forced)."""
    if tiles == "narrow":
        monkeypatch.setenv("INSTANT_SYRK_NARROW", "1")
        monkeypatch.delenv("INSTANT_SYRK_WIDE", raising=False)
    else:
        monkeypatch.setenv("INSTANT_SYRK_WIDE", "1")
        monkeypatch.delenv("INSTANT_SYRK_NARROW", raising=False)


@pytest.mark.parametrize("tiles", ["wide", "narrow"])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("B,L,C", [(2, 64, 64), (3, 300, 200), (4, 49, 448), (2, 256, 1032),
                                   (1, 520, 72), (2, 1000, 136)])
def test_calib_accumulate(torch, monkeypatch, dtype, B, L, C, tiles):
    if dtype == "f32" and tiles == "narrow":
        pytest.skip("one fp32 path")
    _syrk_tiles(monkeypatch, tiles)
    g = rng(500 + L + C)
    t1 = stored(g.standard_normal((B, L, C)), dtype)
    t2 = stored(g.standard_normal((B + 1, L, C)), dtype)
    Cd = torch.zeros(L, L, dtype=torch.float32, device="cuda")
    api = _api()
    api.calib_accumulate(to_dev(t1), Cd)
    api.calib_accumulate(to_dev(t2), Cd)
    torch.cuda.synchronize()
    ref = O.accumulate_autocorrelation(t2, O.accumulate_autocorrelation(t1))
    got = to_np(Cd)
    assert_parity(got, ref, 1e-5 if dtype == "f32" else 1e-4, "C")
    assert np.array_equal(got, got.T) or rel(got, got.T) < 1e-6


@pytest.mark.parametrize("dtype,L,dims", [
    ("bf16", 512, [(32, 768), (32, 3072)]),                    # a layer's C_X and C_G, one launch
    ("bf16", 300, [(3, 200), (5, 264), (2, 64), (4, 136), (1, 8)]),   # five: two launches
    ("bf16", 2048, [(3, 520), (2, 1096)]),                    # channel ranges per tile
    ("bf16", 49, [(40, 448), (40, 1792)]),                    # sample ranges per tile too
    ("f32", 72, [(2, 40), (3, 48)]),
])
@pytest.mark.parametrize("tiles", ["wide", "narrow"])
def test_calib_accumulate_batch(torch, monkeypatch, dtype, L, dims, tiles):
    if dtype == "f32" and tiles == "narrow":
        pytest.skip("one fp32 path")
    _syrk_tiles(monkeypatch, tiles)
    g = rng(700 + L + len(dims))
    ts = [stored(g.standard_normal((B, L, C)), dtype) for B, C in dims]
    api = _api()
    Cb = [torch.zeros(L, L, dtype=torch.float32, device="cuda") for _ in dims]
    Cs = [torch.zeros(L, L, dtype=torch.float32, device="cuda") for _ in dims]
    n0 = api.launch_count()
    api.calib_accumulate_batch([(to_dev(t), C) for t, C in zip(ts, Cb)])
    torch.cuda.synchronize()
    if dtype == "bf16":
        assert api.launch_count() - n0 == (len(dims) + 3) // 4
    for t, C in zip(ts, Cs):
        api.calib_accumulate(to_dev(t), C)
    torch.cuda.synchronize()
    for t, cb, cs in zip(ts, Cb, Cs):
        ref = O.accumulate_autocorrelation(t)
        assert_parity(to_np(cb), ref, 1e-5 if dtype == "f32" else 1e-4, "C (batched)")
        # the same fp32 sums in another order: up to ~sqrt(B * Cdim) * 2^-24 apart
        assert rel(to_np(cb), to_np(cs)) <= 5e-5


def test_device_status_clean(torch):
    assert _api().device_status() == 0


# --------------------------------------------------------------------------
# grad_w_x: both products of the backward in one call
# --------------------------------------------------------------------------
@pytest.mark.parametrize("accumulate", [False, True])
@pytest.mark.parametrize("dtype,B,L,Cx,Cy,Rx,Ry", [
    ("bf16", 32, 512, 768, 768, 8, 8),     # BERT-base block: one launch
    ("bf16", 5, 300, 200, 264, 6, 5),      # ragged g_w tiles (Cy % 128, Cx % 64) in one launch
    ("bf16", 3, 130, 136, 64, 16, 16),     # one K chunk each, a half-filled g_w row tile
    ("bf16", 2, 49, 448, 1792, 8, 8),      # long Cy: two launches
    ("f32", 2, 72, 40, 48, 4, 4),
])
def test_grad_w_x_matches_the_oracle(torch, dtype, B, L, Cx, Cy, Rx, Ry, accumulate):
    api = _api()
    g = rng(1300 + B + L + Cy)
    Sx = stored(g.standard_normal((B * Rx, Cy)), dtype)
    xh = stored(g.standard_normal((B, Rx, Cx)), dtype)
    Sq = stored(g.standard_normal((B * Ry, Cy)), dtype)
    w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), dtype)
    Q = stored(orthonormal_rows(g, Ry, L), dtype)
    gw0 = g.standard_normal((Cy, Cx)).astype(np.float32)
    dt = _tdt(torch, dtype)
    gw = torch.from_numpy(gw0.copy()).cuda() if accumulate else torch.full(
        (Cy, Cx), float("nan"), dtype=torch.float32, device="cuda")
    gx = torch.full((B, L, Cx), float("nan"), dtype=dt, device="cuda")
    ws = torch.empty(max(api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, dt), 16), dtype=torch.uint8,
                     device="cuda")
    api.grad_w_x(to_dev(Sx), to_dev(xh), gw, to_dev(Sq), to_dev(w), to_dev(Q), gx, ws, B,
                 accumulate=accumulate)
    torch.cuda.synchronize()
    ref_w = O.grad_w(O.decode(Sx).reshape(B, Rx, Cy), O.decode(xh))
    if accumulate:
        ref_w = ref_w + gw0.astype(np.float64)
    ref_x = O.grad_x(O.decode(Sq).reshape(B, Ry, Cy), w, Q)
    assert_parity(to_np(gw), ref_w, 1e-5 if dtype == "f32" else 2e-3, "g_w")
    assert_parity(to_np(gx), ref_x, tol(dtype), "g_x")


@pytest.mark.parametrize("kfull", ["0", "1"])
@pytest.mark.parametrize("B,L,Cx,Cy,Rx,Ry", [
    (32, 512, 768, 768, 8, 8),      # BERT-base block: 12 chunks over a cluster of 4
    (6, 384, 200, 520, 4, 16),      # 9 chunks over a cluster of 2, ragged strip
    (4, 1024, 320, 704, 8, 8),      # 11 chunks over a cluster of 8
])
def test_fused_phase_one_whole_or_split(torch, monkeypatch, B, L, Cx, Cy, Rx, Ry, kfull):
    """The single-kernel input gradient with every cluster CTA running the
    whole K of g_hat_x = Sq w (no exchange), or each a slice reduced through
    distributed shared memory: both against the oracle."""
    api = _api()
    monkeypatch.setenv("INSTANT_FUSED_KFULL", kfull)
    g = rng(1400 + B + L + Cy)
    Sx = stored(g.standard_normal((B * Rx, Cy)), "bf16")
    xh = stored(g.standard_normal((B, Rx, Cx)), "bf16")
    Sq = stored(g.standard_normal((B * Ry, Cy)), "bf16")
    w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), "bf16")
    Q = stored(orthonormal_rows(g, Ry, L), "bf16")
    gw = torch.full((Cy, Cx), float("nan"), dtype=torch.float32, device="cuda")
    gx = torch.full((B, L, Cx), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.full((api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, torch.bfloat16),), 255,
                    dtype=torch.uint8, device="cuda")
    n0 = api.launch_count()
    api.grad_w_x(to_dev(Sx), to_dev(xh), gw, to_dev(Sq), to_dev(w), to_dev(Q), gx, ws, B)
    torch.cuda.synchronize()
    assert api.launch_count() - n0 == 1
    ref_w = O.grad_w(O.decode(Sx).reshape(B, Rx, Cy), O.decode(xh))
    ref_x = O.grad_x(O.decode(Sq).reshape(B, Ry, Cy), w, Q)
    assert_parity(to_np(gw), ref_w, 2e-3, "g_w")
    assert_parity(to_np(gx), ref_x, 2e-2, "g_x")
    assert api.device_status() == 0


# --------------------------------------------------------------------------
# grad_w through the write-streaming kernel (short contraction, K = B*Rx <= 256)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("accumulate", [False, True])
@pytest.mark.parametrize("B,Rx,Cx,Cy", [
    (3, 8, 200, 328),       # K = 24: one partial chunk; ragged strip and row tile
    (8, 16, 520, 1000),     # K = 128: two chunks
    (16, 16, 264, 2056),    # K = 256: the largest contraction the kernel takes
    (5, 8, 4104, 1544),     # 845 tiles: CTA ranges cross column strips
    (2, 8, 38400, 128),     # one row tile per strip: x_hat reloaded for every tile
])
def test_grad_w_stream(torch, monkeypatch, B, Rx, Cx, Cy, accumulate):
    monkeypatch.setenv("INSTANT_GRADW_PATH", "stream")
    g = rng(3300 + B + Cx + Cy)
    Sx = stored(g.standard_normal((B * Rx, Cy)), "bf16")
    xh = stored(g.standard_normal((B, Rx, Cx)), "bf16")
    gw0 = g.standard_normal((Cy, Cx)).astype(np.float32)
    gw = to_dev(gw0) if accumulate else nan_like(torch, (Cy, Cx), torch.float32)
    api = _api()
    n0 = api.launch_count()
    api.grad_w(to_dev(Sx), to_dev(xh), gw, B, accumulate=accumulate)
    torch.cuda.synchronize()
    assert api.launch_count() - n0 == 1
    ref = O.grad_w(O.decode(Sx).reshape(B, Rx, Cy), O.decode(xh))
    if accumulate:
        ref = ref + gw0.astype(np.float64)
    assert_parity(to_np(gw), ref, 2e-3, "g_w")
    # the split-K GEMM gives the same products (fp32 sums in another order)
    monkeypatch.setenv("INSTANT_GRADW_PATH", "gemm")
    gw2 = to_dev(gw0) if accumulate else nan_like(torch, (Cy, Cx), torch.float32)
    api.grad_w(to_dev(Sx), to_dev(xh), gw2, B, accumulate=accumulate)
    torch.cuda.synchronize()
    assert_parity(to_np(gw), to_np(gw2), 1e-5, "g_w stream vs gemm")
    assert api.device_status() == 0


# --------------------------------------------------------------------------
# projection with the token axis split across a cluster
# --------------------------------------------------------------------------
@pytest.mark.parametrize("stages", [2, 4])
@pytest.mark.parametrize("split", [2, 3, 4])
@pytest.mark.parametrize("B,L,C,Rx,Ry", [(2, 2048, 392, 16, 16),   # 32 chunks, ragged columns
                                         (3, 1000, 256, 8, 0),     # ragged token tail, compress
                                         (1, 130, 136, 5, 7),      # 3 chunks: short shares
                                         (2, 1024, 264, 32, 32)])  # NT = 64: the largest partials
def test_projection_token_split(torch, monkeypatch, stages, split, B, L, C, Rx, Ry):
    """The token axis split over a 2-4 CTA cluster, with the four-stage and
    the two-stage ring (whose idle ring holds partials up to NT = 64)."""
    monkeypatch.setenv("INSTANT_PROJ_SPLIT", str(split))
    monkeypatch.setenv("INSTANT_PROJ_STAGES", str(stages))
    g = rng(3700 + L + C + split)
    t = stored(g.standard_normal((B, L, C)), "bf16")
    PQ = stored(orthonormal_rows(g, Rx + Ry, L), "bf16")
    api = _api()
    out0 = nan_like(torch, (B * Rx, C), torch.bfloat16)
    if Ry:
        out1 = nan_like(torch, (B * Ry, C), torch.bfloat16)
        api.project_grad(to_dev(t), to_dev(PQ), out0, out1, Rx, Ry)
    else:
        api.compress_act(to_dev(t), to_dev(PQ), out0.view(B, Rx, C))
    torch.cuda.synchronize()
    r0, r1 = O.project_grad(t, PQ[:Rx], PQ[Rx:]) if Ry else (O.compress_act(t, PQ), None)
    assert_parity(to_np(out0).reshape(B, Rx, C), r0, 2e-2, "first plane")
    if Ry:
        assert_parity(to_np(out1).reshape(B, Ry, C), r1, 2e-2, "second plane")
    assert api.device_status() == 0


def test_projection_split_planned_for_the_long_sequence_layer(torch):
    """The plan's own choice on the long-sequence layer's projection (344
    tiles: a 2-CTA token split with the two-stage ring) against the oracle on
    sampled columns of every sample."""
    B, L, C, R = 4, 2048, 11008, 16
    g = rng(3750)
    t = stored(g.standard_normal((B, L, C)) * 0.5, "bf16")
    PQ = stored(orthonormal_rows(g, 2 * R, L), "bf16")
    api = _api()
    Sx = nan_like(torch, (B * R, C), torch.bfloat16)
    Sq = nan_like(torch, (B * R, C), torch.bfloat16)
    api.project_grad(to_dev(t), to_dev(PQ), Sx, Sq, R, R)
    torch.cuda.synchronize()
    cols = np.unique(np.concatenate([np.arange(0, C, 173), [C - 1, 127, 128, 10943]]))
    ts = t[:, :, cols]
    r0, r1 = O.project_grad(ts, PQ[:R], PQ[R:])
    assert_parity(to_np(Sx).reshape(B, R, C)[:, :, cols], r0, 2e-2, "Sx (sampled columns)")
    assert_parity(to_np(Sq).reshape(B, R, C)[:, :, cols], r1, 2e-2, "Sq (sampled columns)")
    assert bool(torch.isfinite(Sx.float()).all()) and bool(torch.isfinite(Sq.float()).all())
    assert api.device_status() == 0


@pytest.mark.parametrize("stages", [2, 4])
@pytest.mark.parametrize("spb", [2, 3, 8])
@pytest.mark.parametrize("B,L,C,Rx,Ry", [(7, 49, 448, 8, 8),     # ViT tokens, a ragged last group
                                         (5, 100, 264, 8, 0),    # compress, two chunks, ragged columns
                                         (3, 128, 136, 64, 64)])  # 128 projector rows, two chunks
def test_projection_samples_per_cta(torch, monkeypatch, stages, spb, B, L, C, Rx, Ry):
    """Several samples per CTA (short token axes), with the two-stage and the
    four-stage ring: against the oracle."""
    monkeypatch.setenv("INSTANT_PROJ_SPB", str(spb))
    monkeypatch.setenv("INSTANT_PROJ_STAGES", str(stages))
    g = rng(3800 + L + C + spb)
    t = stored(g.standard_normal((B, L, C)), "bf16")
    PQ = stored(orthonormal_rows(g, Rx + Ry, L), "bf16")
    api = _api()
    out0 = nan_like(torch, (B * Rx, C), torch.bfloat16)
    if Ry:
        out1 = nan_like(torch, (B * Ry, C), torch.bfloat16)
        api.project_grad(to_dev(t), to_dev(PQ), out0, out1, Rx, Ry)
    else:
        api.compress_act(to_dev(t), to_dev(PQ), out0.view(B, Rx, C))
    torch.cuda.synchronize()
    r0, r1 = O.project_grad(t, PQ[:Rx], PQ[Rx:]) if Ry else (O.compress_act(t, PQ), None)
    assert_parity(to_np(out0).reshape(B, Rx, C), r0, 2e-2, "first plane")
    if Ry:
        assert_parity(to_np(out1).reshape(B, Ry, C), r1, 2e-2, "second plane")
    assert api.device_status() == 0


def test_expand_configurations_in_turn(torch, monkeypatch):
    """Expansions whose shared-memory sizes differ, in the order large, small,
    large again (the second large one plans from cached figures): each still
    launches and matches the oracle."""
    monkeypatch.setenv("INSTANT_EXPAND_BN", "64")
    api = _api()
    for i, (B, L, Cx, Cy, Ry) in enumerate([(4, 512, 256, 64, 16), (6, 49, 192, 64, 16),
                                            (4, 512, 256, 64, 16)]):
        g = rng(3950 + i)
        Sq = stored(g.standard_normal((B * Ry, Cy)), "bf16")
        w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), "bf16")
        Q = stored(orthonormal_rows(g, Ry, L), "bf16")
        gx = nan_like(torch, (B, L, Cx), torch.bfloat16)
        ws = torch.empty((api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, torch.bfloat16),),
                         dtype=torch.uint8, device="cuda")
        api.grad_x_core(to_dev(Sq), to_dev(w), ws, B)
        api.expand(to_dev(Q), gx, ws, Cy)
        torch.cuda.synchronize()
        ref = O.grad_x(O.decode(Sq).reshape(B, Ry, Cy), w, Q)
        assert_parity(to_np(gx), ref, 2e-2, f"g_x, configuration {i}")
    assert api.device_status() == 0


@pytest.mark.parametrize("ctas", [0, 1, 7])  # 0: the planned grid
@pytest.mark.parametrize("bn", [64, 128])
@pytest.mark.parametrize("B,L,Cx,Cy,Ry", [(7, 49, 448, 1792, 8),    # ViT tokens, ragged strips
                                          (5, 300, 264, 136, 16),   # three token tiles per sample
                                          (3, 600, 200, 72, 8),     # five tiles: the Q^T ring (TMA)
                                          (2, 530, 136, 64, 16),    # five tiles, L % 8 != 0: filled ring
                                          (3, 300, 264, 136, 64)])  # Ry = 64: two g_hat_x slots at BN 128
def test_expand_job_runs(torch, monkeypatch, ctas, bn, B, L, Cx, Cy, Ry):
    """The expansion with the (strip, sample, token tile) jobs cut into equal
    runs over a forced grid (one CTA takes every job; runs starting inside a
    sample or a strip) and both strip widths, against the oracle."""
    if ctas:
        monkeypatch.setenv("INSTANT_EXPAND_CTAS", str(ctas))
    monkeypatch.setenv("INSTANT_EXPAND_BN", str(bn))
    api = _api()
    g = rng(3900 + L + Cx + Ry + ctas + bn)
    Sq = stored(g.standard_normal((B * Ry, Cy)), "bf16")
    w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), "bf16")
    Q = stored(orthonormal_rows(g, Ry, L), "bf16")
    gx = nan_like(torch, (B, L, Cx), torch.bfloat16)
    ws = torch.full((api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, torch.bfloat16),), 255,
                    dtype=torch.uint8, device="cuda")
    api.grad_x_core(to_dev(Sq), to_dev(w), ws, B)
    api.expand(to_dev(Q), gx, ws, Cy)
    torch.cuda.synchronize()
    ref = O.grad_x(O.decode(Sq).reshape(B, Ry, Cy), w, Q)
    assert_parity(to_np(gx), ref, 2e-2, "g_x")
    assert api.device_status() == 0


@pytest.mark.parametrize("splits", [0, 1, 3, 5, 7, 8])  # 0: the planned split
@pytest.mark.parametrize("long_a", [False, True])
@pytest.mark.parametrize("B,Ry,Cx,Cy", [(4, 16, 1096, 1000),  # M = 64: the 64-row A box, ragged K
                                        (3, 8, 264, 520),     # M = 24
                                        (5, 16, 200, 456)])   # M = 80: the 128-row box
def test_grad_x_core_splits(torch, monkeypatch, splits, long_a, B, Ry, Cx, Cy):
    """g_hat_x = Sq w from the split-K GEMM with K cut into 1..8 cluster shares
    (including uneven ones) and either A box, read from the workspace (filled
    with NaN first) and compared element by element with the oracle."""
    if splits:
        monkeypatch.setenv("INSTANT_GEMM_SPLITS", str(splits))
    if long_a:
        monkeypatch.setenv("INSTANT_GEMM_LONG_A", "1")
    api = _api()
    g = rng(4100 + B + Ry + Cx + Cy + splits)
    Sq = stored(g.standard_normal((B * Ry, Cy)), "bf16")
    w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), "bf16")
    n = api.grad_x_workspace_bytes(B, 130, Cx, Cy, Ry, torch.bfloat16)
    assert n == B * Ry * Cx * 2
    ws = torch.full((n,), 255, dtype=torch.uint8, device="cuda")
    api.grad_x_core(to_dev(Sq), to_dev(w), ws, B)
    torch.cuda.synchronize()
    got = to_np(ws.view(torch.bfloat16).reshape(B, Ry, Cx))
    ref = O.grad_x_core(O.decode(Sq).reshape(B, Ry, Cy), w)
    assert_parity(got, ref, 2e-2, "g_hat_x")
    assert api.device_status() == 0


def test_grad_x_core_planned_for_the_long_sequence_layer(torch):
    """The plan's own choice for the long-sequence layer's g_hat_x = Sq w
    (64 rows, K = 11008: the 64-row A box, K split over a cluster) against
    the oracle on sampled columns; every element written and finite."""
    B, Ry, Cx, Cy = 4, 16, 4096, 11008
    g = rng(4200)
    Sq = stored(g.standard_normal((B * Ry, Cy)), "bf16")
    w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), "bf16")
    api = _api()
    ws = torch.full((api.grad_x_workspace_bytes(B, 2048, Cx, Cy, Ry, torch.bfloat16),), 255,
                    dtype=torch.uint8, device="cuda")
    api.grad_x_core(to_dev(Sq), to_dev(w), ws, B)
    torch.cuda.synchronize()
    got = ws.view(torch.bfloat16).reshape(B, Ry, Cx)
    assert bool(torch.isfinite(got.float()).all())
    cols = np.unique(np.concatenate([np.arange(0, Cx, 37), [63, 64, 4032, Cx - 1]]))
    ref = O.grad_x_core(O.decode(Sq).reshape(B, Ry, Cy), O.decode(w)[:, cols])
    assert_parity(to_np(got)[:, :, cols], ref, 2e-2, "g_hat_x (sampled columns)")
    assert api.device_status() == 0
