"""Calibration solve on the GPU against the oracle's eigendecomposition.

Inputs are autocorrelation sums with planted spectra (built on the host), so
k and R are known to be decided with margin; k and R must match exactly."""

import numpy as np
import pytest

import oracle as O
from gpu_util import orthonormal_rows, rel, rng, to_dev, to_np, torch_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


def _planted_C(seed, L, lam, n, noise=0.0):
    g = rng(seed)
    U = orthonormal_rows(g, L, L).T
    C = (U * lam[None, :]) @ U.T
    if noise:
        N = g.standard_normal((L, L)) * noise
        C = C + 0.5 * (N + N.T)
    return (C * n).astype(np.float32)


def _margin(lam, E, eps):
    cum = np.cumsum(np.asarray(lam) ** 2)
    return float(np.min(np.abs(cum - eps * E)) / E)


def _check(torch, C_sum, n, *, eps, p, r_override, scale_on, r_cap, out_dtype):
    from rank_compressed_backprop_gb300 import api

    L = C_sum.shape[0]
    rows = torch.empty(r_cap, L, dtype=out_dtype, device="cuda")
    res = api.calib_solve(to_dev(C_sum), n, rows, eps=eps, p=p, r_override=r_override,
                          scale_on=scale_on)
    ref = O.calibrate(C_sum.astype(np.float64), n, eps=eps, p=p, r_override=r_override,
                      scale_on=scale_on)
    assert _margin(ref["eigenvalues"], ref["energy"], eps) > 1e-4, "case decided without margin"
    assert res.k == ref["k"]
    assert res.R == ref["R"]
    assert abs(res.energy - ref["energy"]) <= 1e-9 * ref["energy"]
    R = ref["R"]
    got_eig = np.array(res.eigenvalues[:R])
    assert rel(got_eig, ref["eigenvalues"][:R]) <= 1e-4
    assert abs(res.scale - ref["scale"]) <= 1e-4 * ref["scale"]
    got = to_np(rows)
    assert np.all(got[R:] == 0)
    # rows are s * u_i^T with canonical signs; compare scale-free
    g1 = got[:R] / ref["scale"]
    r1 = ref["rows"] / ref["scale"]
    lim = 2e-3 if out_dtype == torch.float32 else 1.5e-2
    assert np.max(np.abs(g1 - r1)) <= lim
    return res, ref


@pytest.mark.parametrize("L", [16, 49, 64, 100, 128])
def test_jacobi_path_planted(torch, L):
    lam = 1e3 * np.arange(1, L + 1, dtype=np.float64) ** -2.0
    C = _planted_C(10 + L, L, lam, n=8)
    _check(torch, C, 8, eps=0.95, p=2, r_override=0, scale_on=True, r_cap=min(L, 16),
           out_dtype=torch.float32)


@pytest.mark.parametrize("L", [129, 300, 512])
def test_subspace_path_planted(torch, L):
    lam = 1e5 * np.arange(1, L + 1, dtype=np.float64) ** -3.0 + 7.0
    C = _planted_C(20 + L, L, lam, n=64)
    _check(torch, C, 64, eps=0.95, p=2, r_override=8, scale_on=True, r_cap=8,
           out_dtype=torch.bfloat16)
    _check(torch, C, 64, eps=0.95, p=2, r_override=0, scale_on=False, r_cap=16,
           out_dtype=torch.float32)


def test_subspace_long_sequence(torch):
    # long-sequence statistic (L = 2048, sigma_i ~ i^-1, lambda ~ i^-2 plus a noise floor)
    L = 2048
    lam = 5e6 * np.arange(1, L + 1, dtype=np.float64) ** -2.0 + 41.0
    C = _planted_C(31, L, lam, n=64)
    _check(torch, C, 64, eps=0.95, p=4, r_override=16, scale_on=True, r_cap=16,
           out_dtype=torch.bfloat16)


def test_flat_tail_needs_more_rank(torch):
    # energy spread over many modes: k near 20 forces a larger block (L > 128)
    L = 256
    lam = np.concatenate([np.full(20, 10.0) * np.linspace(1.0, 0.6, 20), np.full(L - 20, 0.05)])
    C = _planted_C(41, L, lam, n=4)
    _check(torch, C, 4, eps=0.9, p=2, r_override=0, scale_on=True, r_cap=32,
           out_dtype=torch.float32)


def test_warm_start_reproduces_the_cold_solve(torch):
    from rank_compressed_backprop_gb300 import api

    L = 512
    lam = 1e5 * np.arange(1, L + 1, dtype=np.float64) ** -3.0 + 7.0
    C = to_dev(_planted_C(77, L, lam, n=64))
    cold = torch.empty(8, L, dtype=torch.bfloat16, device="cuda")
    r0 = api.calib_solve(C, 64, cold, eps=0.95, p=2, r_override=8)
    warm = cold.clone()
    r1 = api.calib_solve(C, 64, warm, eps=0.95, p=2, r_override=8, warm_start=True)
    assert (r1.k, r1.R) == (r0.k, r0.R)
    assert abs(r1.scale - r0.scale) <= 1e-5 * r0.scale
    assert float((warm.float() - cold.float()).abs().max()) <= 2e-2 * float(cold.float().abs().max())
    # a warm start from an unrelated projector still converges to the same answer
    other = torch.randn(8, L, device="cuda").to(torch.bfloat16)
    r2 = api.calib_solve(C, 64, other, eps=0.95, p=2, r_override=8, warm_start=True)
    assert (r2.k, r2.R) == (r0.k, r0.R)
    assert float((other.float() - cold.float()).abs().max()) <= 2e-2 * float(cold.float().abs().max())


@pytest.mark.parametrize("path", ["one_launch", "multi_launch"])
@pytest.mark.parametrize("L", [200, 512])
def test_mid_size_solvers_match_the_oracle(torch, monkeypatch, path, L):
    """Both solvers for 128 < L <= 512 -- the whole iteration in one cluster
    launch, and the multi-launch host loop -- against the oracle."""
    if path == "multi_launch":
        monkeypatch.setenv("INSTANT_SOLVER_MULTI", "1")
    lam = 2e4 * np.arange(1, L + 1, dtype=np.float64) ** -2.5 + 3.0
    C = _planted_C(60 + L, L, lam, n=32)
    _check(torch, C, 32, eps=0.95, p=2, r_override=16, scale_on=True, r_cap=16,
           out_dtype=torch.bfloat16)
    _check(torch, C, 32, eps=0.9, p=3, r_override=0, scale_on=True, r_cap=24,
           out_dtype=torch.float32)


def test_block_too_short_hands_over_to_a_larger_block(torch):
    # k + p beyond the first block (32 columns): the one-launch solve stops and
    # the multi-launch loop carries on with 64 columns
    L = 300
    lam = np.concatenate([np.linspace(10.0, 6.0, 40), np.full(L - 40, 0.02)])
    C = _planted_C(43, L, lam, n=4)
    res, ref = _check(torch, C, 4, eps=0.9, p=2, r_override=0, scale_on=True, r_cap=48,
                      out_dtype=torch.float32)
    assert res.R > 31


def test_one_launch_solver_rejects_bad_statistics(torch):
    from rank_compressed_backprop_gb300 import api
    from rank_compressed_backprop_gb300._lib import InstantError

    L = 300
    rows = torch.full((8, L), 5.0, dtype=torch.float32, device="cuda")
    for C in (torch.zeros(L, L, device="cuda"), torch.eye(L, device="cuda")):
        if C[0, 0] == 1:
            C[7, 11] = float("nan")
        with pytest.raises(InstantError) as e:
            api.calib_solve(C, 4, rows, r_override=8)
        assert e.value.status == 8
        assert bool((rows == 5.0).all())   # nothing written
    assert api.device_status() == 0


@pytest.mark.parametrize("r_override", [8, 16])
def test_mid_size_solve_converges_in_one_launch(torch, r_override):
    """For 128 < L <= 512 and blocks of 16 or 32 columns the whole solve is one
    cluster launch: no hand-over to the multi-launch loop on a planted spectrum."""
    from rank_compressed_backprop_gb300 import api

    L = 512
    lam = 1e5 * np.arange(1, L + 1, dtype=np.float64) ** -2.0 + 5.0
    C = to_dev(_planted_C(88, L, lam, n=64))
    rows = torch.empty(r_override, L, dtype=torch.bfloat16, device="cuda")
    n0 = api.launch_count()
    res = api.calib_solve(C, 64, rows, eps=0.95, p=2, r_override=r_override)
    assert api.launch_count() - n0 == 1
    assert res.R == r_override
    n0 = api.launch_count()
    api.calib_solve(C, 64, rows, eps=0.95, p=2, r_override=r_override, warm_start=True)
    assert api.launch_count() - n0 == 1


@pytest.mark.parametrize("path", ["one_launch", "multi_launch"])
@pytest.mark.parametrize("L", [1024, 1500, 2048])
def test_long_solvers_match_the_oracle(torch, monkeypatch, path, L):
    """512 < L <= 2048: the one-launch cluster solve with the basis exchanged
    through the workspace (each CTA keeps only its own rows), and the
    multi-launch loop, against the oracle; 1500 tokens leave the last CTA a
    shorter share of rows."""
    if path == "multi_launch":
        monkeypatch.setenv("INSTANT_SOLVER_MULTI", "1")
    lam = 5e6 * np.arange(1, L + 1, dtype=np.float64) ** -2.0 + 41.0
    C = _planted_C(90 + L, L, lam, n=64)
    _check(torch, C, 64, eps=0.95, p=4, r_override=16, scale_on=True, r_cap=16,
           out_dtype=torch.bfloat16)
    _check(torch, C, 64, eps=0.95, p=2, r_override=8, scale_on=False, r_cap=8,
           out_dtype=torch.float32)


@pytest.mark.parametrize("r_override", [8, 16])
def test_long_solve_converges_in_one_launch(torch, r_override):
    from rank_compressed_backprop_gb300 import api

    L = 2048
    lam = 5e6 * np.arange(1, L + 1, dtype=np.float64) ** -2.0 + 41.0
    C = to_dev(_planted_C(95, L, lam, n=64))
    rows = torch.empty(r_override, L, dtype=torch.bfloat16, device="cuda")
    n0 = api.launch_count()
    res = api.calib_solve(C, 64, rows, eps=0.95, p=4, r_override=r_override)
    assert api.launch_count() - n0 == 1
    assert res.R == r_override
    n0 = api.launch_count()
    api.calib_solve(C, 64, rows, eps=0.95, p=4, r_override=r_override, warm_start=True)
    assert api.launch_count() - n0 == 1
    assert api.device_status() == 0
