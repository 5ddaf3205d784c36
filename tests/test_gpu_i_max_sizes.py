"""The largest token length the calibration accepts (L = 8192): the
accumulation against entries of the oracle computed one by one, and the solve
against a planted spectrum whose eigenvectors are known in closed form
(a Householder basis U = I - 2 v v^T, so C = U diag(lam) U^T costs O(L^2))."""

import numpy as np
import pytest

import oracle as O
from gpu_util import rng, stored, to_dev, to_np, torch_or_skip

pytestmark = pytest.mark.gpu

L_MAX = 8192


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


def test_accumulate_at_the_largest_token_length(torch):
    from rank_compressed_backprop_gb300 import api

    g = rng(8100)
    B, Cd = 2, 16
    t = stored(g.standard_normal((B, L_MAX, Cd)), "bf16")
    C = torch.zeros(L_MAX, L_MAX, dtype=torch.float32, device="cuda")
    api.calib_accumulate(to_dev(t), C)
    torch.cuda.synchronize()
    td = O.decode(t)
    ii = g.integers(0, L_MAX, 3000)
    jj = g.integers(0, L_MAX, 3000)
    # sampled entries one by one, plus the diagonal blocks' corners
    ii = np.concatenate([ii, [0, L_MAX - 1, 8191, 4095]])
    jj = np.concatenate([jj, [L_MAX - 1, 0, 8191, 4096]])
    got = C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()].double().cpu().numpy()
    want = np.einsum("bic,bic->i", td[:, ii, :], td[:, jj, :])
    scale = np.sqrt(np.einsum("bic,bic->i", td[:, ii, :], td[:, ii, :])
                    * np.einsum("bic,bic->i", td[:, jj, :], td[:, jj, :]))
    # fp32 dot product of B * Cd = 32 terms: |error| <= 32 * 2^-24 * scale
    assert np.max(np.abs(got - want) / scale) <= 4e-6
    assert api.device_status() == 0


def test_solve_at_the_largest_token_length(torch):
    from rank_compressed_backprop_gb300 import api

    g = rng(8200)
    v = g.standard_normal(L_MAX)
    v /= np.linalg.norm(v)
    lam = np.full(L_MAX, 0.01)
    lam[:12] = [100.0, 80.0, 64.0, 51.0, 41.0, 33.0, 26.0, 21.0, 5.0, 4.0, 3.0, 2.0]
    n = 16
    # C = U diag(lam) U^T with U = I - 2 v v^T, formed in O(L^2)
    lv = lam * v
    C = np.diag(lam) - 2.0 * np.outer(v, lv) - 2.0 * np.outer(lv, v) + 4.0 * float(v @ lv) * np.outer(v, v)
    E = float(np.sum(lam ** 2))
    eps, p, R = 0.95, 2, 8
    k = O.truncation_index(lam, E, eps)
    cum = np.cumsum(lam ** 2)
    assert np.min(np.abs(cum - eps * E)) / E > 1e-3   # k decided with margin
    rows = torch.empty(R, L_MAX, dtype=torch.bfloat16, device="cuda")
    Cd = torch.from_numpy((C * n).astype(np.float32)).cuda()
    del C
    res = api.calib_solve(Cd, n, rows, eps=eps, p=p, r_override=R)
    assert (res.k, res.R) == (k, R)
    assert abs(res.energy - E) <= 1e-6 * E
    got_eig = np.array(res.eigenvalues[:R])
    assert np.max(np.abs(got_eig - lam[:R]) / lam[:R]) <= 1e-4
    s = 1.0 / np.sqrt(np.sum(lam[:R] ** 2))
    assert abs(res.scale - s) <= 1e-4 * s
    got = to_np(rows) / s
    for i in range(R):
        u = -2.0 * v[i] * v
        u[i] += 1.0                       # u_i = e_i - 2 v_i v: largest entry at i, positive
        assert np.max(np.abs(got[i] - u)) <= 1.5e-2
    assert api.device_status() == 0
