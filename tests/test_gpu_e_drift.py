"""Reconstruction error under subspace drift (the oversampling study): the
CUDA reconstruction-error kernel against a float64 restatement of its sum,
and the whole drift loop against the oracle on the drifting ViT-MLP workload."""

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import orthonormal_rows, rng, stored, to_dev, torch_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


@pytest.mark.parametrize("dtype,B,L,C,R", [("bf16", 3, 49, 1792, 8), ("bf16", 2, 130, 264, 5),
                                           ("f32", 2, 33, 40, 3), ("f32", 1, 7, 13, 1)])
def test_reconstruction_error_kernel(torch, dtype, B, L, C, R):
    from rank_compressed_backprop_gb300 import api

    g = rng(1700 + B + L + C)
    t = stored(g.standard_normal((B, L, C)), dtype)
    Q = stored(orthonormal_rows(g, R, L), dtype)
    td, Qd = O.decode(t), O.decode(Q)
    S = stored(np.einsum("rl,blc->brc", Qd, td), dtype)
    Sd = O.decode(S)
    rec = np.einsum("rl,brc->blc", Qd, Sd)
    want_e2 = float(((td - rec) ** 2).sum())
    want_n2 = float((td ** 2).sum())
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    e2, n2 = api.reconstruction_error(to_dev(t), to_dev(Q), to_dev(S).view(B * R, C), ws)
    assert abs(n2 - want_n2) <= 1e-5 * want_n2
    assert abs(e2 - want_e2) <= 1e-4 * want_e2 + 1e-7 * want_n2


@pytest.mark.parametrize("p,n_t", [(0, 2), (4, 100)])
def test_drift_loop_matches_the_oracle(torch, p, n_t):
    from rank_compressed_backprop_gb300.drift import drift_errors

    wl = W.workload("vit_mlp_pair_49")
    li = W.LayerInputs(wl)          # first layer: g_y [256, 49, 1792], planted rank-6 spectrum
    steps = 4
    host = [li.g_y(t) for t in range(steps)]
    run = drift_errors(lambda t: to_dev(host[t]), steps, n_t, p, eps=wl.eps)
    # the same loop in the oracle: statistic of the step's batch, unscaled
    # projector with oversampling p, reconstruction error of the step's batch
    rows = None
    for t in range(steps):
        if t % n_t == 0:
            C = O.accumulate_autocorrelation(host[t])
            cal = O.calibrate(C, host[t].shape[0], eps=wl.eps, p=p, r_override=0, scale_on=False)
            rows = cal["rows"]
            got = [c for c in run.calibrations if c[0] == t][0]
            assert (got[1], got[2]) == (cal["k"], cal["R"])
        want = O.reconstruction_error(host[t], rows)
        assert abs(run.errors[t] - want) <= 1e-2 * max(want, 0.05), (t, run.errors[t], want)
    if n_t > steps:
        # no recalibration after step 0: the error can only grow with the drift
        assert run.errors[-1] > run.errors[0]
