"""Layer driver, CUDA-graph capture, checkpoint/resume and failure paths."""

import io
import os

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import assert_parity, rel, stored, to_dev, to_np, torch_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


def _layer_inputs(B=4, L=136, Cx=264, Cy=200):
    U = W.planted_basis(3, L, L)
    x = W.planted_batch(4, U, W.sigma_profile("power", L, L, Cx, True, 1.5), B, Cx, 0.1, False)
    g = W.planted_batch(5, U, W.sigma_profile("power", L, L, Cy, True, 1.5), B, Cy, 0.1, False)
    w = W.weight(6, Cy, Cx, 0.02)
    return stored(x, "bf16"), stored(g, "bf16"), stored(w, "bf16")


def _make_layer(torch, w, B, L, R=8):
    from rank_compressed_backprop_gb300 import InstantLinear

    return InstantLinear(to_dev(w), B=B, L=L, Rx=R, Ry=R, n_t=3, eps=0.95, p=2)


def test_layer_step_schedule_and_oracle(torch):
    x, g, w = _layer_inputs()
    B, L = x.shape[0], x.shape[1]
    lay = _make_layer(torch, w, B, L)
    xd, gd = to_dev(x), to_dev(g)
    for t in range(4):
        gw, gx = lay.step(xd, gd)
        if t == 0:
            rx, rg = lay.last_calibration
            cx = O.calibrate(O.accumulate_autocorrelation(x), B, eps=0.95, p=2, r_override=8)
            assert rx.k == cx["k"]
    torch.cuda.synchronize()
    assert lay.t == 4 and lay.n_x == 0
    # the per-step outputs equal the oracle's given the layer's current projector
    P = lay.P.view(torch.int16).cpu().numpy().view(np.uint16)
    Q = lay.Q.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = O.low_rank_backward(x, g, w, P, Q)
    assert_parity(to_np(gw), ref["g_w"], 2e-2, "g_w")
    assert_parity(to_np(gx), ref["g_x"], 2e-2, "g_x")


@pytest.mark.parametrize("L", [49, 136])
def test_layers_recalibrated_together(torch, L):
    """LayerCalibration solves several layers' statistics in one call: given
    the same statistics (copied: the accumulation adds with atomics, so two
    accumulations may differ in their last bits), each layer's projector, k and
    R bit for bit as its own recalibrate gives them, cold and warm-started,
    and the statistics are cleared."""
    from rank_compressed_backprop_gb300 import LayerCalibration

    x, g, w = _layer_inputs(L=L)
    x2, g2, w2 = _layer_inputs(L=L, Cx=200, Cy=264)
    B = x.shape[0]
    pairs = [(x, g, w), (x2, g2, w2)]
    alone = [_make_layer(torch, ww, B, L) for _, _, ww in pairs]
    together = [_make_layer(torch, ww, B, L) for _, _, ww in pairs]
    cal = LayerCalibration(together)
    for rnd in range(2):  # cold, then warm-started
        want = []
        for a, b, (xx, gg, _) in zip(alone, together, pairs):
            a.accumulate(to_dev(xx), to_dev(gg))
            b.C_X.copy_(a.C_X)
            b.C_G.copy_(a.C_G)
            b.n_x, b.n_g = a.n_x, a.n_g
            want.append(a.recalibrate())
        got = cal.recalibrate()
        torch.cuda.synchronize()
        for a, b, (ra, rb) in zip(alone, together, zip(want, got)):
            assert torch.equal(a.PQ, b.PQ), rnd
            assert (ra[0].k, ra[0].R, ra[1].k, ra[1].R) == (rb[0].k, rb[0].R, rb[1].k, rb[1].R)
            assert b.n_x == 0 and int(b.C_X.count_nonzero()) == 0 and int(b.C_G.count_nonzero()) == 0


def test_cuda_graph_replay_matches_eager(torch):
    x, g, w = _layer_inputs()
    B, L = x.shape[0], x.shape[1]
    lay = _make_layer(torch, w, B, L)
    xd, gd = to_dev(x), to_dev(g)
    lay.accumulate(xd, gd)
    lay.recalibrate()
    lay.compress(xd)
    gw, gx = lay.backward(gd)
    torch.cuda.synchronize()
    gw_e, gx_e = gw.clone(), gx.clone()
    gw.zero_()
    gx.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            lay.compress(xd)
            lay.backward(gd)
    torch.cuda.current_stream().wait_stream(s)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(gw, gw_e)
    assert torch.equal(gx, gx_e)


def test_checkpoint_resume_identical(torch):
    x, g, w = _layer_inputs()
    B, L = x.shape[0], x.shape[1]
    a = _make_layer(torch, w, B, L)
    xd, gd = to_dev(x), to_dev(g)
    a.step(xd, gd)
    a.accumulate(xd, gd)   # a half-accumulated statistic is part of the state
    buf = io.BytesIO()
    torch.save({"PQ": a.PQ, "C_X": a.C_X, "C_G": a.C_G, "n_x": a.n_x, "n_g": a.n_g, "t": a.t}, buf)
    buf.seek(0)
    st = torch.load(buf)
    b = _make_layer(torch, w, B, L)
    b.PQ.copy_(st["PQ"])
    b.C_X.copy_(st["C_X"])
    b.C_G.copy_(st["C_G"])
    b.n_x, b.n_g, b.t = st["n_x"], st["n_g"], st["t"]
    ga = [t.clone() for t in a.step(xd, gd)]
    gb = [t.clone() for t in b.step(xd, gd)]
    torch.cuda.synchronize()
    assert torch.equal(ga[0], gb[0]) and torch.equal(ga[1], gb[1])


def test_solver_failure_paths(torch, monkeypatch):
    from rank_compressed_backprop_gb300 import api
    from rank_compressed_backprop_gb300._lib import InstantError

    rows = torch.empty(4, 64, dtype=torch.float32, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(InstantError) as e:
        api.calib_solve(C, 4, rows)
    assert e.value.status == 8   # zero energy
    C = torch.eye(64, dtype=torch.float32, device="cuda")
    C[3, 5] = float("nan")
    with pytest.raises(InstantError) as e:
        api.calib_solve(C, 4, rows)
    assert e.value.status == 8   # non-finite
    # forced iteration caps (host-side fault injection)
    g = np.random.Generator(np.random.PCG64(1))
    for L in (64, 300):
        A = g.standard_normal((L, L))
        Cg = to_dev((A @ A.T).astype(np.float32))
        rows = torch.empty(8, L, dtype=torch.float32, device="cuda")
        monkeypatch.setenv("INSTANT_FAULT", "solve_noconv")
        _, st = api.calib_solve(Cg, 1, rows, r_override=8, raise_on_error=False)
        assert st == 7
        monkeypatch.delenv("INSTANT_FAULT")
    # the context is healthy afterwards and no device-side wait ran out
    assert api.device_status() == 0
    y = torch.ones(8, device="cuda") * 2
    assert float(y.sum()) == 16.0


def test_bad_arguments_raise_before_launch(torch):
    from rank_compressed_backprop_gb300 import api

    x = torch.zeros(1, 64, 60, dtype=torch.bfloat16, device="cuda")  # Cx not a multiple of 8
    P = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    xh = torch.zeros(1, 4, 60, dtype=torch.bfloat16, device="cuda")
    from rank_compressed_backprop_gb300._lib import InstantError

    with pytest.raises(InstantError) as e:
        api.compress_act(x, P, xh)
    assert e.value.status == 4
    assert api.device_status() == 0
