"""instant_forward: y = x w^T with x_hat = P x formed from the same staged x
tiles, against the oracle's forward and compression (INSTANT page, overall
framework), on ragged shapes, the fallback shapes and the long-sequence
layer."""

import numpy as np
import pytest

import oracle as O
from gpu_util import (assert_parity, nan_like, orthonormal_rows, rng, stored, to_dev, to_np, tol,
                      torch_or_skip)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


def _api():
    from rank_compressed_backprop_gb300 import api

    return api


def _tdt(torch, dtype):
    return torch.float32 if dtype == "f32" else torch.bfloat16


def _run(torch, dtype, B, L, Cx, Cy, Rx, seed):
    api = _api()
    g = rng(seed)
    x = stored(g.standard_normal((B, L, Cx)), dtype)
    w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cx), dtype)
    P = stored(orthonormal_rows(g, Rx, L), dtype) if Rx else None
    dt = _tdt(torch, dtype)
    y = nan_like(torch, (B, L, Cy), dt)
    xh = nan_like(torch, (B, Rx, Cx), dt) if Rx else None
    ws = api.forward_workspace(B, L, Cx, Rx, dt, "cuda")
    n0 = api.launch_count()
    api.forward(to_dev(x), to_dev(w), y, to_dev(P) if Rx else None, xh, ws if Rx else None)
    torch.cuda.synchronize()
    launches = api.launch_count() - n0
    return x, w, P, y, xh, ws, launches


@pytest.mark.parametrize("dtype,B,L,Cx,Cy,Rx,fused", [
    ("bf16", 2, 256, 512, 768, 8, True),       # two token tiles per sample, four column tiles
    ("bf16", 3, 384, 256, 200, 16, True),      # column tail (200 % 192)
    ("bf16", 1, 128, 4096, 392, 32, True),     # the largest fused rank, 64 channel chunks
    ("bf16", 32, 512, 768, 768, 8, True),      # the BERT-base block's layer (B = 32, L = 512)
    ("bf16", 2, 256, 264, 200, 16, False),     # 264 channels: no chunk pairs -> two launches
    ("bf16", 2, 130, 256, 384, 8, False),      # 130 tokens: tiles straddle samples -> two launches
    ("bf16", 2, 256, 512, 384, 40, False),     # rank beyond the flush warp -> two launches
    ("bf16", 3, 256, 520, 200, 0, None),       # y only
    ("f32", 2, 72, 40, 48, 4, False),
])
def test_forward_matches_the_oracle(torch, dtype, B, L, Cx, Cy, Rx, fused):
    x, w, P, y, xh, ws, launches = _run(torch, dtype, B, L, Cx, Cy, Rx, 4100 + L + Cx + Rx)
    assert_parity(to_np(y), O.forward(x, w), tol(dtype), "y")
    if Rx:
        assert_parity(to_np(xh), O.compress_act(x, P), tol(dtype), "x_hat")
        # the workspace (fp32 partial sums and counters) is zero again
        assert int(ws.count_nonzero()) == 0
    if fused is True:
        assert launches == 1
    elif fused is False:
        assert launches == 2
    assert _api().device_status() == 0


def test_repeated_calls_reuse_the_workspace(torch):
    """Three calls in a row on one workspace, the second with other inputs:
    each gives the result of its own inputs -- y bit for bit the same for the
    same inputs; x_hat's fp32 partial sums are added with atomics, so its
    rounding may differ in the last bit between calls."""
    api = _api()
    B, L, Cx, Cy, Rx = 2, 512, 768, 768, 8
    outs = []
    for seed in (4200, 4201, 4200):
        g = rng(seed)
        x = to_dev(stored(g.standard_normal((B, L, Cx)), "bf16"))
        w = to_dev(stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cx), "bf16"))
        P = to_dev(stored(orthonormal_rows(g, Rx, L), "bf16"))
        outs.append((x, w, P))
    ws = api.forward_workspace(B, L, Cx, Rx, torch.bfloat16, "cuda")
    res = []
    for x, w, P in outs:
        y = nan_like(torch, (B, L, Cy), torch.bfloat16)
        xh = nan_like(torch, (B, Rx, Cx), torch.bfloat16)
        api.forward(x, w, y, P, xh, ws)
        res.append((y, xh))
    torch.cuda.synchronize()
    assert torch.equal(res[0][0], res[2][0])
    assert_parity(to_np(res[2][1]), to_np(res[0][1]), 1e-2, "x_hat, same inputs again")
    assert not torch.equal(res[0][1], res[1][1])
    for (x, _, P), (_, xh) in zip(outs, res):
        assert_parity(to_np(xh), O.compress_act(x.view(torch.int16).cpu().numpy().view(np.uint16),
                                                P.view(torch.int16).cpu().numpy().view(np.uint16)),
                      2e-2, "x_hat")
    assert int(ws.count_nonzero()) == 0


def test_fused_and_separate_x_hat_agree(torch, monkeypatch):
    """x_hat from the GEMM's staged tiles and from the projection kernel: the
    same fp32 sums in another order, rounded once to bf16."""
    B, L, Cx, Cy, Rx = 2, 384, 640, 400, 16
    _, _, _, y1, xh1, _, n1 = _run(torch, "bf16", B, L, Cx, Cy, Rx, 4300)
    monkeypatch.setenv("INSTANT_NO_FUSED_FORWARD", "1")
    _, _, _, y2, xh2, _, n2 = _run(torch, "bf16", B, L, Cx, Cy, Rx, 4300)
    assert (n1, n2) == (1, 2)
    assert torch.equal(y1, y2)
    assert_parity(to_np(xh1), to_np(xh2), 1e-2, "x_hat fused vs separate")


def test_forward_long_sequence_layer(torch):
    """The long-sequence 4096 -> 11008 layer (B = 4, L = 2048, Rx = 16) on its
    seeded inputs and the oracle's projector."""
    import workloads as W

    api = _api()
    wl = W.workload("long_seq_4096_11008")
    li = W.LayerInputs(wl)
    x, w = li.x(), li.w()
    P = stored(orthonormal_rows(rng(4400), wl.Rx, wl.L), "bf16")
    B, L, Cx, Cy, Rx = wl.B, wl.L, li.Cx, li.Cy, wl.Rx
    y = nan_like(torch, (B, L, Cy), torch.bfloat16)
    xh = nan_like(torch, (B, Rx, Cx), torch.bfloat16)
    ws = api.forward_workspace(B, L, Cx, Rx, torch.bfloat16, "cuda")
    api.forward(to_dev(x), to_dev(w), y, to_dev(P), xh, ws)
    torch.cuda.synchronize()
    assert_parity(to_np(y), O.forward(x, w), 2e-2, "y")
    assert_parity(to_np(xh), O.compress_act(x, P), 2e-2, "x_hat")
    assert int(ws.count_nonzero()) == 0
    assert api.device_status() == 0


def test_layer_forward_keeps_x_hat_for_the_backward(torch):
    """InstantLinear.forward returns y and leaves x_hat = P x where the
    backward reads it: the backward after forward equals the backward after
    compress."""
    from rank_compressed_backprop_gb300 import InstantLinear

    import workloads as W

    # planted decaying spectra, so that the energy rule's k + p fits the solver's block
    B, L, Cx, Cy, R = 2, 256, 384, 512, 8
    U = W.planted_basis(45, L, L)
    x = to_dev(stored(W.planted_batch(46, U, W.sigma_profile("power", L, L, Cx, True, 1.5), B, Cx,
                                      0.1, False), "bf16"))
    gy = to_dev(stored(W.planted_batch(47, U, W.sigma_profile("power", L, L, Cy, True, 1.5), B, Cy,
                                       0.1, False), "bf16"))
    w = to_dev(stored(rng(4500).standard_normal((Cy, Cx)) / np.sqrt(Cx), "bf16"))
    lay = InstantLinear(w, B=B, L=L, Rx=R, Ry=R, n_t=10)
    lay.accumulate(x, gy)
    lay.recalibrate()
    y = lay.forward(x)
    torch.cuda.synchronize()
    assert_parity(to_np(y), O.forward(x.view(torch.int16).cpu().numpy().view(np.uint16),
                                      w.view(torch.int16).cpu().numpy().view(np.uint16)),
                  2e-2, "y")
    xh_fwd = lay.xhat.clone()
    gw1, gx1 = [t.clone() for t in lay.backward(gy)]
    lay.compress(x)
    torch.cuda.synchronize()
    assert_parity(to_np(xh_fwd), to_np(lay.xhat), 1e-2, "x_hat forward vs compress")
    gw2, gx2 = lay.backward(gy)
    torch.cuda.synchronize()
    assert_parity(to_np(gw1), to_np(gw2), 2e-2, "g_w")
    assert_parity(to_np(gx1), to_np(gx2), 2e-2, "g_x")
