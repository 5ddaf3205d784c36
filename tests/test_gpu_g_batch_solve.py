"""instant_calib_solve_batch: every problem gets what a call of
instant_calib_solve on it alone gives (bit for bit where the one-launch solver
runs), whichever solver path it takes, and the problems that the one-launch
solver takes share its launches."""

import numpy as np
import pytest

import oracle as O
from gpu_util import orthonormal_rows, rel, rng, to_dev, to_np, torch_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


def _planted(seed, L, lam, n):
    g = rng(seed)
    U = orthonormal_rows(g, L, L).T
    return ((U * lam[None, :]) @ U.T * n).astype(np.float32)


def _spectrum(L, a, s, floor):
    return a * np.arange(1, L + 1, dtype=np.float64) ** -s + floor


def _solve_both(torch, specs, dtype):
    """specs: (C_host, n, r_cap, params) -> batch results, single results, rows."""
    from rank_compressed_backprop_gb300 import api

    L = specs[0][0].shape[0]
    Cs = [to_dev(c) for c, _, _, _ in specs]
    seed_rows = [torch.randn(r, L, device="cuda").to(dtype) for _, _, r, _ in specs]
    rows_b = [s.clone() for s in seed_rows]
    rows_s = [s.clone() for s in seed_rows]
    probs = [dict(C=C, n_samples=n, rows_out=rb, **prm)
             for C, rb, (_, n, _, prm) in zip(Cs, rows_b, specs)]
    res_b = api.calib_solve_batch(probs)
    res_s = [api.calib_solve(C, n, rs, **prm) for C, rs, (_, n, _, prm) in zip(Cs, rows_s, specs)]
    return res_b, res_s, rows_b, rows_s


def _same(res_b, res_s, rows_b, rows_s, torch, exact=None):
    """Bit for bit where the one-launch solver ran (exact[i]); elsewhere the
    multi-launch path adds some partial sums with atomics, so two runs of it
    agree up to that rounding order."""
    for i, (a, b, ra, rb) in enumerate(zip(res_b, res_s, rows_b, rows_s)):
        assert (a.k, a.R) == (b.k, b.R)
        if exact is None or exact[i]:
            assert (a.scale, a.energy) == (b.scale, b.energy)
            assert a.eigenvalues == b.eigenvalues
            assert torch.equal(ra, rb)
        else:
            assert abs(a.scale - b.scale) <= 1e-6 * abs(b.scale)
            assert abs(a.energy - b.energy) <= 1e-9 * b.energy
            assert rel(np.array(a.eigenvalues[: a.R]), np.array(b.eigenvalues[: b.R])) <= 1e-6
            d = float((ra.float() - rb.float()).abs().max())
            assert d <= 1e-4 * float(rb.float().abs().max())


def test_pair_is_one_launch_and_matches_two_solves(torch):
    from rank_compressed_backprop_gb300 import api

    L = 512
    specs = [(_planted(301, L, _spectrum(L, 1e5, 3.0, 7.0), 64), 64, 8,
              dict(eps=0.95, p=2, r_override=8)),
             (_planted(302, L, _spectrum(L, 3e4, 2.0, 1.0), 64), 64, 8,
              dict(eps=0.95, p=2, r_override=8, warm_start=True))]
    n0 = api.launch_count()
    res_b, res_s, rows_b, rows_s = _solve_both(torch, specs, torch.bfloat16)
    # one launch for the batch, one per single solve
    assert api.launch_count() - n0 == 3
    _same(res_b, res_s, rows_b, rows_s, torch)
    for (C, n, _, prm), r, rows in zip(specs, res_b, rows_b):
        ref = O.calibrate(C.astype(np.float64), n, eps=prm["eps"], p=prm["p"],
                          r_override=prm["r_override"])
        assert (r.k, r.R) == (ref["k"], ref["R"])
        assert rel(np.array(r.eigenvalues[:r.R]), ref["eigenvalues"][:r.R]) <= 1e-4
        got = to_np(rows)[: r.R] / ref["scale"]
        assert np.max(np.abs(got - ref["rows"] / ref["scale"])) <= 1.5e-2
    assert api.device_status() == 0


def test_mixed_paths_match_single_solves(torch):
    """Blocks of 16 and 32 columns (two launches), a block that proves too
    short and hands over to the multi-launch loop, all in one call."""
    L = 300
    short = np.concatenate([np.linspace(10.0, 6.0, 40), np.full(L - 40, 0.02)])
    specs = [(_planted(311, L, _spectrum(L, 2e4, 2.5, 3.0), 32), 32, 16,
              dict(eps=0.95, p=2, r_override=16)),          # block of 32
             (_planted(312, L, _spectrum(L, 2e4, 2.5, 3.0), 32), 32, 24,
              dict(eps=0.9, p=3, r_override=0)),            # block of 16
             (_planted(313, L, short, 4), 4, 48, dict(eps=0.9, p=2, r_override=0)),  # too short
             (_planted(314, L, _spectrum(L, 5e3, 2.0, 1.0), 16), 16, 8,
              dict(eps=0.95, p=2, r_override=8))]
    res_b, res_s, rows_b, rows_s = _solve_both(torch, specs, torch.float32)
    _same(res_b, res_s, rows_b, rows_s, torch, exact=[True, True, False, True])
    assert res_b[2].R > 31


def test_small_and_many(torch):
    """L <= 128 (full Jacobi) and more problems than one launch holds."""
    from rank_compressed_backprop_gb300 import api

    specs = [(_planted(320 + i, 96, _spectrum(96, 1e3, 2.0, 0.5), 8), 8, 8,
              dict(eps=0.95, p=1, r_override=0)) for i in range(3)]
    res_b, res_s, rows_b, rows_s = _solve_both(torch, specs, torch.float32)
    _same(res_b, res_s, rows_b, rows_s, torch, exact=[False] * 3)
    L = 256
    specs = [(_planted(340 + i, L, _spectrum(L, 1e4, 2.0 + 0.05 * i, 1.0), 16), 16, 8,
              dict(eps=0.95, p=2, r_override=8)) for i in range(17)]
    n0 = api.launch_count()
    res_b, res_s, rows_b, rows_s = _solve_both(torch, specs, torch.bfloat16)
    assert api.launch_count() - n0 == 2 + 17     # 16 + 1 clusters, then one per single solve
    _same(res_b, res_s, rows_b, rows_s, torch)


def test_bad_problem_stops_the_whole_call(torch):
    from rank_compressed_backprop_gb300 import api

    L = 256
    C = to_dev(_planted(350, L, _spectrum(L, 1e4, 2.0, 1.0), 16))
    good = torch.full((8, L), 3.0, device="cuda")
    bad = torch.full((8, L), 3.0, device="cuda")
    n0 = api.launch_count()
    res, st = api.calib_solve_batch([dict(C=C, n_samples=16, rows_out=good, r_override=8),
                                     dict(C=C, n_samples=16, rows_out=bad, r_override=9)],
                                    raise_on_error=False)
    assert st == [2, 2]                       # INSTANT_ERR_SHAPE everywhere
    assert api.launch_count() == n0
    assert bool((good == 3.0).all()) and bool((bad == 3.0).all())
    # a statistic without energy fails alone; the other is solved
    Z = torch.zeros(L, L, device="cuda")
    res, st = api.calib_solve_batch([dict(C=C, n_samples=16, rows_out=good, r_override=8),
                                     dict(C=Z, n_samples=16, rows_out=bad, r_override=8)],
                                    raise_on_error=False)
    assert st == [0, 8]
    assert res[0].R == 8 and not bool((good == 3.0).all())
    assert api.device_status() == 0


@pytest.mark.parametrize("L", [49, 100, 128])
def test_small_statistics_in_one_synchronisation(torch, L):
    """L <= 128 (full Jacobi): the batch queues every problem's launches and
    reads all results with one synchronisation; each result is bit for bit
    the single call's, and a statistic without energy fails alone, its rows
    untouched."""
    from rank_compressed_backprop_gb300 import api

    specs = [(_planted(360 + L + i, L, _spectrum(L, 1e4, 1.5 + 0.5 * i, 1.0), 32), 32, 8,
              dict(eps=0.95, p=2, r_override=0)) for i in range(3)]
    res_b, res_s, rows_b, rows_s = _solve_both(torch, specs, torch.bfloat16)
    _same(res_b, res_s, rows_b, rows_s, torch)
    for r in res_b:
        assert r.R >= 1
    C = to_dev(specs[0][0])
    good = torch.full((8, L), 3.0, device="cuda")
    bad = torch.full((8, L), 3.0, device="cuda")
    Z = torch.zeros(L, L, device="cuda")
    res, st = api.calib_solve_batch([dict(C=C, n_samples=32, rows_out=good, r_override=8),
                                     dict(C=Z, n_samples=32, rows_out=bad, r_override=8)],
                                    raise_on_error=False)
    assert st == [0, 8]
    assert res[0].R == 8 and not bool((good == 3.0).all())
    assert bool((bad == 3.0).all())
    assert api.device_status() == 0
