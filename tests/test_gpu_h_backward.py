"""instant_backward: the projection of g_y and both gradients in one call (one
launch where the single-kernel input gradient applies), against the oracle
and, bit for bit, against the two separate calls it replaces."""

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


def _inputs(g, dtype, B, L, Cx, Cy, Rx, Ry):
    gy = stored(g.standard_normal((B, L, Cy)), dtype)
    xh = stored(g.standard_normal((B, Rx, Cx)), dtype)
    w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), dtype)
    PQ = stored(np.concatenate([orthonormal_rows(g, Rx, L), orthonormal_rows(g, Ry, L)]), dtype)
    return gy, xh, w, PQ


def _run(torch, api, dtype, B, L, Cx, Cy, Rx, Ry, gy, xh, w, PQ, ws, gw0=None, fused=True):
    dt = _tdt(torch, dtype)
    Sx = torch.full((B * Rx, Cy), float("nan"), dtype=dt, device="cuda")
    Sq = torch.full((B * Ry, Cy), float("nan"), dtype=dt, device="cuda")
    gw = (torch.from_numpy(gw0.copy()).cuda() if gw0 is not None
          else torch.full((Cy, Cx), float("nan"), dtype=torch.float32, device="cuda"))
    gx = torch.full((B, L, Cx), float("nan"), dtype=dt, device="cuda")
    n0 = api.launch_count()
    if fused:
        api.backward(gy, PQ, xh, w, Sx, Sq, gw, gx, ws, Rx, accumulate=gw0 is not None)
    else:
        ws2 = torch.empty(max(api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, dt), 16),
                          dtype=torch.uint8, device="cuda")
        api.project_grad(gy, PQ, Sx, Sq, Rx, Ry)
        api.grad_w_x(Sx, xh, gw, Sq, w, PQ[Rx:], gx, ws2, B, accumulate=gw0 is not None)
    torch.cuda.synchronize()
    return Sx, Sq, gw, gx, api.launch_count() - n0


CASES = [
    # dtype, B, L, Cx, Cy, Rx, Ry, one launch (None: whatever fits)
    ("bf16", 32, 512, 768, 768, 8, 8, True),      # BERT-base block
    ("bf16", 5, 300, 200, 264, 6, 5, True),       # ragged tiles everywhere
    ("bf16", 3, 130, 136, 64, 16, 16, True),      # one projection tile per sample
    ("bf16", 4, 49, 256, 384, 8, 8, True),        # L % 8 != 0: the projector filled by threads
    ("bf16", 64, 256, 512, 768, 4, 4, None),      # more tiles than CTAs in a group
    ("bf16", 2, 49, 448, 1792, 8, 8, False),      # long Cy: projection, then grad_w_x
    ("f32", 2, 72, 40, 48, 4, 4, False),
]


@pytest.mark.parametrize("one_launch", [False, True])
@pytest.mark.parametrize("accumulate", [False, True])
@pytest.mark.parametrize("dtype,B,L,Cx,Cy,Rx,Ry,launches", CASES)
def test_backward_matches_oracle_and_separate_calls(torch, monkeypatch, dtype, B, L, Cx, Cy, Rx, Ry,
                                                    launches, accumulate, one_launch):
    from rank_compressed_backprop_gb300 import api

    if one_launch:
        monkeypatch.setenv("INSTANT_ONE_LAUNCH_BACKWARD", "1")
    else:
        monkeypatch.delenv("INSTANT_ONE_LAUNCH_BACKWARD", raising=False)
        launches = False

    g = rng(1500 + B + L + Cy + Rx)
    gy, xh, w, PQ = _inputs(g, dtype, B, L, Cx, Cy, Rx, Ry)
    dt = _tdt(torch, dtype)
    ws = api.backward_workspace(B, L, Cx, Cy, Ry, dt, "cuda")
    gw0 = g.standard_normal((Cy, Cx)).astype(np.float32) if accumulate else None
    d = [to_dev(a) for a in (gy, xh, w, PQ)]
    Sx, Sq, gw, gx, n = _run(torch, api, dtype, B, L, Cx, Cy, Rx, Ry, *d, ws, gw0)
    # the counters are back at zero after the call
    assert int(ws[:(B + 3) * 4].count_nonzero()) == 0
    # oracle
    P, Q = O.decode(PQ)[:Rx], O.decode(PQ)[Rx:]
    ref_sx, ref_sq = O.project_grad(gy, P, Q)
    ref_w = O.grad_w(ref_sx, O.decode(xh))
    if accumulate:
        ref_w = ref_w + gw0.astype(np.float64)
    ref_x = O.grad_x(ref_sq, w, Q)
    assert_parity(to_np(Sx).reshape(ref_sx.shape), ref_sx, tol(dtype), "Sx")
    assert_parity(to_np(Sq).reshape(ref_sq.shape), ref_sq, tol(dtype), "Sq")
    assert_parity(to_np(gw), ref_w, 1e-5 if dtype == "f32" else 2e-2, "g_w")
    assert_parity(to_np(gx), ref_x, tol(dtype), "g_x")
    # bit for bit what project_grad + grad_w_x give
    Sx2, Sq2, gw2, gx2, n2 = _run(torch, api, dtype, B, L, Cx, Cy, Rx, Ry, *d, ws, gw0, fused=False)
    for a, b in ((Sx, Sx2), (Sq, Sq2), (gw, gw2), (gx, gx2)):
        assert torch.equal(a, b)
    if launches is True:
        assert n == 1
    elif launches is False:
        assert n == n2
    else:
        assert n in (1, n2)
    assert api.device_status() == 0


def test_back_to_back_calls_and_graph_replay(torch, monkeypatch):
    """One launch: the counters reset themselves, so calls in a row, and
    replays of a CUDA graph holding several calls, each give the result of
    their own inputs."""
    from rank_compressed_backprop_gb300 import api

    monkeypatch.setenv("INSTANT_ONE_LAUNCH_BACKWARD", "1")

    dtype, B, L, Cx, Cy, Rx, Ry = "bf16", 32, 512, 768, 768, 8, 8
    dt = torch.bfloat16
    ws = api.backward_workspace(B, L, Cx, Cy, Ry, dt, "cuda")
    sets = []
    for k in range(3):
        g = rng(1600 + k)
        d = [to_dev(a) for a in _inputs(g, dtype, B, L, Cx, Cy, Rx, Ry)]
        outs = (nan_like(torch, (B * Rx, Cy), dt), nan_like(torch, (B * Ry, Cy), dt),
                nan_like(torch, (Cy, Cx), torch.float32), nan_like(torch, (B, L, Cx), dt))
        sets.append((d, outs))
    ref = []
    for d, _ in sets:
        Sx, Sq, gw, gx, _ = _run(torch, api, dtype, B, L, Cx, Cy, Rx, Ry, *d, ws, fused=False)
        ref.append((Sx, Sq, gw, gx))

    def call(k):
        (gy, xh, w, PQ), (Sx, Sq, gw, gx) = sets[k]
        api.backward(gy, PQ, xh, w, Sx, Sq, gw, gx, ws, Rx)

    for rep in range(2):
        for k in range(3):
            call(k)
    torch.cuda.synchronize()
    for (_, outs), r in zip(sets, ref):
        for a, b in zip(outs, r):
            assert torch.equal(a, b)
    for _, outs in sets:
        for t in outs:
            t.zero_()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cs):
        with torch.cuda.graph(graph, stream=cs):
            for k in (0, 1, 2, 1):
                call(k)
    torch.cuda.current_stream().wait_stream(cs)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for (_, outs), r in zip(sets, ref):
        for a, b in zip(outs, r):
            assert torch.equal(a, b)
    assert int(ws.count_nonzero()) == 0 or int(ws[:(B + 3) * 4].count_nonzero()) == 0
    assert api.device_status() == 0
