"""Pins of the fp64 oracle against what the INSTANT page and the mathematics fix.

Every check here is independent of the oracle's own formulas: closed forms
printed on the page, hand-worked cases, identities that hold exactly for
special inputs, and scalar brute force on tiny inputs.  A dropped term, a
wrong operand or a transposed product in the oracle fails at least one.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(s):
    return np.random.Generator(np.random.PCG64(s))


def _orthonormal_rows(rng, R, L):
    q, _ = np.linalg.qr(rng.standard_normal((L, R)))
    return q.T


# --------------------------------------------------------------------------
# T1: FLOP closed forms (关键设计 3)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L,Cx,Cy,Rx,Ry", [(7, 5, 3, 2, 1), (16, 12, 20, 4, 3),
                                           (49, 24, 40, 8, 8), (64, 64, 64, 4, 4)])
def test_flop_tally_matches_closed_forms(L, Cx, Cy, Rx, Ry):
    rng = _rng(1)
    x = rng.standard_normal((1, L, Cx))
    g = rng.standard_normal((1, L, Cy))
    w = rng.standard_normal((Cy, Cx))
    P = rng.standard_normal((Rx, L))
    Q = rng.standard_normal((Ry, L))
    t = O.FlopTally()
    O.low_rank_backward(x, g, w, P, Q, tally=t)
    assert t.flops == 2 * (Rx + Ry) * (Cx * Cy + L * Cx + L * Cy)
    assert t.flops == O.flops_low_rank(L, Cx, Cy, Rx, Ry)
    tv = O.FlopTally()
    O.vanilla_backward(x, g, w, tally=tv)
    assert tv.flops == 4 * L * Cx * Cy == O.flops_vanilla(L, Cx, Cy)


def test_flop_tally_scales_with_batch():
    rng = _rng(2)
    B, L, Cx, Cy, R = 3, 10, 6, 8, 2
    t = O.FlopTally()
    O.low_rank_backward(rng.standard_normal((B, L, Cx)), rng.standard_normal((B, L, Cy)),
                        rng.standard_normal((Cy, Cx)), rng.standard_normal((R, L)),
                        rng.standard_normal((R, L)), tally=t)
    assert t.flops == B * O.flops_low_rank(L, Cx, Cy, R, R)


def test_bert_block_saving_matches_page():
    g = json.load(open(os.path.join(GOLDEN, "bert_block_flops.json")))
    v = O.flops_vanilla(g["L"], g["Cx"], g["Cy"])
    lr = O.flops_low_rank(g["L"], g["Cx"], g["Cy"], g["Rx"], g["Ry"])
    assert v == 1_207_959_552 and lr == 44_040_192
    ratio = v / lr
    assert abs(ratio - g["printed_saving"]) < 0.5
    assert abs(ratio - 27.4286) < 1e-3


# --------------------------------------------------------------------------
# T2: identity -- full orthonormal P, Q (R = L) give the vanilla gradients
# --------------------------------------------------------------------------
@pytest.mark.parametrize("kind", ["identity", "random"])
def test_full_rank_orthonormal_projection_is_vanilla(kind):
    rng = _rng(3)
    B, L, Cx, Cy = 3, 12, 9, 7
    x = rng.standard_normal((B, L, Cx))
    g = rng.standard_normal((B, L, Cy))
    w = rng.standard_normal((Cy, Cx))
    if kind == "identity":
        P = np.eye(L)
        Q = np.eye(L)
    else:
        P = _orthonormal_rows(rng, L, L)
        Q = _orthonormal_rows(rng, L, L)
    lr = O.low_rank_backward(x, g, w, P, Q)
    # vanilla by scalar loops (independent of the oracle's products)
    gw = np.zeros((Cy, Cx))
    gx = np.zeros((B, L, Cx))
    for b in range(B):
        for i in range(Cy):
            for j in range(Cx):
                gw[i, j] += sum(g[b, l, i] * x[b, l, j] for l in range(L))
        for l in range(L):
            for j in range(Cx):
                gx[b, l, j] = sum(g[b, l, i] * w[i, j] for i in range(Cy))
    assert np.allclose(lr["g_w"], gw, rtol=1e-12, atol=1e-12)
    assert np.allclose(lr["g_x"], gx, rtol=1e-12, atol=1e-12)
    van = O.vanilla_backward(x, g, w)
    assert np.allclose(van["g_w"], gw, rtol=1e-12, atol=1e-12)
    assert np.allclose(van["g_x"], gx, rtol=1e-12, atol=1e-12)


def test_partial_rank_is_not_vanilla():
    # guards the identity test: with R < L on generic data the two differ
    rng = _rng(4)
    B, L, Cx, Cy = 2, 10, 5, 6
    x, g = rng.standard_normal((B, L, Cx)), rng.standard_normal((B, L, Cy))
    w = rng.standard_normal((Cy, Cx))
    P = _orthonormal_rows(rng, 3, L)
    lr = O.low_rank_backward(x, g, w, P, P)
    van = O.vanilla_backward(x, g, w)
    assert np.linalg.norm(lr["g_w"] - van["g_w"]) > 1e-3 * np.linalg.norm(van["g_w"])


# --------------------------------------------------------------------------
# brute force of each product on tiny inputs
# --------------------------------------------------------------------------
def test_products_by_scalar_loops():
    rng = _rng(5)
    B, L, Cx, Cy, Rx, Ry = 2, 5, 3, 4, 2, 3
    x = rng.standard_normal((B, L, Cx))
    g = rng.standard_normal((B, L, Cy))
    w = rng.standard_normal((Cy, Cx))
    P = rng.standard_normal((Rx, L))
    Q = rng.standard_normal((Ry, L))
    r = O.low_rank_backward(x, g, w, P, Q)
    for b in range(B):
        for i in range(Rx):
            for c in range(Cx):
                assert math.isclose(r["x_hat"][b, i, c],
                                    sum(P[i, l] * x[b, l, c] for l in range(L)), rel_tol=1e-12)
            for c in range(Cy):
                assert math.isclose(r["Sx"][b, i, c],
                                    sum(P[i, l] * g[b, l, c] for l in range(L)), rel_tol=1e-12)
        for i in range(Ry):
            for c in range(Cy):
                assert math.isclose(r["Sq"][b, i, c],
                                    sum(Q[i, l] * g[b, l, c] for l in range(L)), rel_tol=1e-12)
            for c in range(Cx):
                assert math.isclose(r["gx_hat"][b, i, c],
                                    sum(r["Sq"][b, i, k] * w[k, c] for k in range(Cy)),
                                    rel_tol=1e-12)
        for l in range(L):
            for c in range(Cx):
                assert math.isclose(r["g_x"][b, l, c],
                                    sum(Q[i, l] * r["gx_hat"][b, i, c] for i in range(Ry)),
                                    rel_tol=1e-11, abs_tol=1e-13)
    for cy in range(Cy):
        for cx in range(Cx):
            ref = sum(r["Sx"][b, i, cy] * r["x_hat"][b, i, cx] for b in range(B) for i in range(Rx))
            assert math.isclose(r["g_w"][cy, cx], ref, rel_tol=1e-11, abs_tol=1e-13)


def test_accumulate_by_scalar_loops_and_additivity():
    rng = _rng(6)
    t = rng.standard_normal((3, 4, 5))
    C = O.accumulate_autocorrelation(t)
    for i in range(4):
        for j in range(4):
            ref = sum(t[b, i, c] * t[b, j, c] for b in range(3) for c in range(5))
            assert math.isclose(C[i, j], ref, rel_tol=1e-12)
    C1 = O.accumulate_autocorrelation(t[:1])
    C12 = O.accumulate_autocorrelation(t[1:], C1)
    assert np.allclose(C12, C, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# T3: planted rank-k inputs are reconstructed exactly
# --------------------------------------------------------------------------
def _planted_exact(rng, B, L, C, d):
    """t_b = U diag(d) O_b with orthonormal U [L,k] and O_b [k,C] (O O^T = I)."""
    k = len(d)
    U = _orthonormal_rows(rng, k, L).T
    out = np.empty((B, L, C))
    for b in range(B):
        Ob = _orthonormal_rows(rng, k, C)
        out[b] = U @ np.diag(d) @ Ob
    return out, U


def test_planted_rank_k_projection_recovers_vanilla():
    rng = _rng(7)
    B, L, Cx, Cy = 4, 16, 10, 12
    x, Ux = _planted_exact(rng, B, L, Cx, [3.0, 2.0, 1.0])
    g, Ug = _planted_exact(rng, B, L, Cy, [5.0, 0.5])
    w = rng.standard_normal((Cy, Cx))
    lr = O.low_rank_backward(x, g, w, Ux.T, Ug.T)
    van = O.vanilla_backward(x, g, w)
    assert np.allclose(lr["g_w"], van["g_w"], rtol=1e-11, atol=1e-11)
    assert np.allclose(lr["g_x"], van["g_x"], rtol=1e-11, atol=1e-11)


def test_calibrated_projection_on_planted_data_and_scale_closed_form():
    rng = _rng(8)
    B, L, Cx, Cy = 6, 16, 10, 12
    dx = np.array([3.0, 2.0, 1.0])
    dg = np.array([5.0, 0.5])
    x, _ = _planted_exact(rng, B, L, Cx, dx)
    g, _ = _planted_exact(rng, B, L, Cy, dg)
    w = rng.standard_normal((Cy, Cx))
    Cxs = O.accumulate_autocorrelation(x)
    Cgs = O.accumulate_autocorrelation(g)
    # every sample has x_b x_b^T = U diag(d^2) U^T, so E[x x^T] has eigenvalues d^2
    cx = O.calibrate(Cxs, B, eps=0.95, p=0, r_override=3, scale_on=False)
    cg = O.calibrate(Cgs, B, eps=0.95, p=0, r_override=2, scale_on=False)
    assert np.allclose(cx["eigenvalues"][:3], dx ** 2, rtol=1e-12)
    lr = O.low_rank_backward(x, g, w, cx["rows"], cg["rows"])
    van = O.vanilla_backward(x, g, w)
    assert np.allclose(lr["g_w"], van["g_w"], rtol=1e-10, atol=1e-10)
    assert np.allclose(lr["g_x"], van["g_x"], rtol=1e-10, atol=1e-10)
    # scale on: s = (sum_{i<=R} (d_i^2)^2)^(-1/2); g_w carries s_P^2, g_x carries s_Q^2
    sx = (np.sum(dx ** 4)) ** -0.5
    sg = (np.sum(dg ** 4)) ** -0.5
    cx1 = O.calibrate(Cxs, B, eps=0.95, p=0, r_override=3, scale_on=True)
    cg1 = O.calibrate(Cgs, B, eps=0.95, p=0, r_override=2, scale_on=True)
    assert math.isclose(cx1["scale"], sx, rel_tol=1e-12)
    assert math.isclose(cg1["scale"], sg, rel_tol=1e-12)
    lr1 = O.low_rank_backward(x, g, w, cx1["rows"], cg1["rows"])
    assert np.allclose(lr1["g_w"], sx ** 2 * van["g_w"], rtol=1e-10, atol=1e-12)
    assert np.allclose(lr1["g_x"], sg ** 2 * van["g_x"], rtol=1e-10, atol=1e-12)
    # energy: E = ||C||_F^2 = sum d^4 ; with eps=0.95 on d=(3,2,1): 81/98 < .95, 97/98 >= .95
    assert math.isclose(cx["energy"], float(np.sum(dx ** 4)), rel_tol=1e-12)
    assert cx["k"] == 2
    # d=(5, .5): 625/625.0625 >= .95 -> k = 1
    assert cg["k"] == 1


# --------------------------------------------------------------------------
# T4: truncation index
# --------------------------------------------------------------------------
def test_truncation_hand_cases():
    cases = json.load(open(os.path.join(GOLDEN, "truncation_cases.json")))["cases"]
    for c in cases:
        lam = np.array(c["sigma"], np.float64)
        E = float(np.sum(lam * lam))
        assert O.truncation_index(lam, E, c["eps"]) == c["k"], c


def test_truncation_via_calibrate_on_planted_spectrum():
    rng = _rng(9)
    for L in (3, 5, 8):
        for trial in range(20):
            lam = np.sort(rng.uniform(0.01, 1.0, L))[::-1]
            U = _orthonormal_rows(rng, L, L).T
            C = U @ np.diag(lam) @ U.T
            eps = float(rng.uniform(0.3, 0.99))
            # brute force over all candidate k, from the known spectrum
            E = float(np.sum(lam ** 2))
            cands = [k for k in range(1, L + 1) if np.sum(lam[:k] ** 2) >= eps * E]
            k_ref = min(cands)
            margin = min(abs(np.sum(lam[:k] ** 2) - eps * E) for k in range(1, L + 1)) / E
            if margin < 1e-9:
                continue
            for p in (0, 1, 2, L):
                out = O.calibrate(C, 1, eps=eps, p=p, scale_on=False)
                assert out["k"] == k_ref
                assert out["R"] == min(k_ref + p, L)


def test_calibrate_rejects_zero_energy():
    with pytest.raises(FloatingPointError):
        O.calibrate(np.zeros((4, 4)), 3)


# --------------------------------------------------------------------------
# T5: eigensolver -- planted spectra and exact invariants
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L", [2, 3, 6, 17, 64])
def test_eig_recovers_planted_spectrum(L):
    rng = _rng(10 + L)
    lam = np.sort(rng.uniform(0.1, 10.0, L))[::-1]
    U = _orthonormal_rows(rng, L, L).T
    C = U @ np.diag(lam) @ U.T
    got, V = O.eig_desc(C)
    assert np.allclose(got, lam, rtol=1e-11, atol=1e-11)
    R = max(1, L // 2)
    assert np.allclose(V[:, :R] @ V[:, :R].T, U[:, :R] @ U[:, :R].T, atol=1e-9)
    # residuals and invariants (trace, Frobenius, determinant)
    assert np.allclose(C @ V, V * got[None, :], atol=1e-10)
    assert math.isclose(np.trace(C), got.sum(), rel_tol=1e-12)
    assert math.isclose(O.frobenius_energy(C), float(np.sum(got ** 2)), rel_tol=1e-12)
    if L <= 6:
        assert math.isclose(np.linalg.det(C), float(np.prod(got)), rel_tol=1e-9)


def test_eig_descending_and_canonical_sign():
    rng = _rng(11)
    A = rng.standard_normal((7, 7))
    C = A @ A.T
    lam, V = O.eig_desc(C)
    assert np.all(np.diff(lam) <= 0)
    Vc = O.canonical_sign(V)
    for j in range(7):
        i = int(np.argmax(np.abs(Vc[:, j])))
        assert Vc[i, j] > 0
        assert np.allclose(np.abs(Vc[:, j]), np.abs(V[:, j]))


def test_calibrate_rank_clamp_and_override():
    rng = _rng(12)
    L = 6
    U = _orthonormal_rows(rng, L, L).T
    lam = np.array([10.0, 9.0, 8.0, 7.0, 6.0, 5.0])
    C = U @ np.diag(lam) @ U.T
    out = O.calibrate(C, 1, eps=0.95, p=100, scale_on=False)
    assert out["R"] == L
    out2 = O.calibrate(C, 1, eps=0.95, p=0, r_override=2, scale_on=False)
    assert out2["R"] == 2 and out2["rows"].shape == (2, L)
    assert np.allclose(out2["rows"] @ out2["rows"].T, np.eye(2), atol=1e-12)


# --------------------------------------------------------------------------
# T6: sign invariance -- outputs depend on P^T P and Q^T Q only
# --------------------------------------------------------------------------
def test_sign_flip_invariance():
    rng = _rng(13)
    B, L, Cx, Cy, R = 3, 11, 6, 5, 4
    x, g = rng.standard_normal((B, L, Cx)), rng.standard_normal((B, L, Cy))
    w = rng.standard_normal((Cy, Cx))
    P = _orthonormal_rows(rng, R, L)
    Q = _orthonormal_rows(rng, R, L)
    D = np.diag([1.0, -1.0, -1.0, 1.0])
    a = O.low_rank_backward(x, g, w, P, Q)
    b = O.low_rank_backward(x, g, w, D @ P, D @ Q)
    assert np.allclose(a["g_w"], b["g_w"], rtol=1e-12, atol=1e-12)
    assert np.allclose(a["g_x"], b["g_x"], rtol=1e-12, atol=1e-12)


def test_reconstruction_error_limits():
    rng = _rng(14)
    L = 9
    t = rng.standard_normal((2, L, 4))
    assert O.reconstruction_error(t, np.eye(L)) < 1e-12
    V = _orthonormal_rows(rng, 3, L)
    e = O.reconstruction_error(t, V)
    assert 0.0 < e < 1.0


def test_decode_bf16_bits():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x7F7F], np.uint16)
    vals = O.decode(bits)
    assert vals[0] == 1.0 and vals[1] == -1.0 and vals[3] == 0.0
    assert vals[2] == 3.140625
    assert vals[4] == 2.0 ** 127 * (255.0 / 128.0)


def test_reconstruction_error_hand_worked_values():
    """Exact values worked out by hand (INSTANT page, 关键设计 2: the fraction of
    the gradient that the rank-R projector loses).  Each case is chosen so that
    a plausible slip gives another number: the squared ratio (no square root),
    a per-sample mean instead of the pooled Frobenius ratio, a normalisation by
    ||t||^2, or the projector applied the wrong way round."""
    L, C = 9, 2
    V = np.eye(L)[:3]                       # keeps tokens 0, 1, 2
    t = np.zeros((1, L, C))
    t[0, 0, 0] = 2.0
    t[0, 1, 1] = 2.0
    t[0, 2, 0] = 2.0
    t[0, 2, 1] = 2.0                        # kept energy 16
    t[0, 5, 1] = 3.0                        # lost energy 9
    e = O.reconstruction_error(t, V)
    assert abs(e - 0.6) < 1e-15             # 3 / 5; the square would be 0.36
    # a second sample that the projector keeps whole: pooled 3/7, not the
    # per-sample mean (0.6 + 0) / 2 = 0.3
    t2 = np.zeros((2, L, C))
    t2[0] = t[0]
    t2[1, 0, 0], t2[1, 1, 0], t2[1, 2, 1] = 4.0, 2.0, 2.0      # energy 24, all kept
    assert abs(O.reconstruction_error(t2, V) - 3.0 / 7.0) < 1e-15
    # one row that is not an axis: v = (0.6, 0.8, 0); t = (1, 0, 0) projects to
    # 0.6 v = (0.36, 0.48, 0), leaving (0.64, -0.48, 0) of norm 0.8
    v = np.array([[0.6, 0.8, 0.0]])
    assert abs(O.reconstruction_error(np.array([[[1.0], [0.0], [0.0]]]), v) - 0.8) < 1e-15
    # (3, 4, 5): (3, 4) lies on v, 5 is lost: 5 / sqrt(50)
    got = O.reconstruction_error(np.array([[[3.0], [4.0], [5.0]]]), v)
    assert abs(got - 5.0 / np.sqrt(50.0)) < 1e-15
    # a vector orthogonal to v is lost whole, one on v is kept whole
    assert abs(O.reconstruction_error(np.array([[[4.0], [-3.0], [0.0]]]), v) - 1.0) < 1e-15
    assert O.reconstruction_error(np.array([[[3.0], [4.0], [0.0]]]), v) < 1e-15


def test_reconstruction_error_planted_closed_form():
    """t = V^T a + n with n orthogonal to the rows of V: the error is
    ||n|| / sqrt(||a||^2 + ||n||^2) exactly (the two parts are orthogonal)."""
    rng = _rng(15)
    B, L, C, R = 3, 40, 7, 5
    Qf, _ = np.linalg.qr(rng.standard_normal((L, L)))
    V = Qf[:, :R].T                         # orthonormal rows
    W = Qf[:, R:]                           # basis of the orthogonal complement
    a = rng.standard_normal((B, R, C))
    n = 0.3 * rng.standard_normal((B, L - R, C))
    t = V.T[None] @ a + W[None] @ n
    want = np.sqrt(np.sum(n * n)) / np.sqrt(np.sum(a * a) + np.sum(n * n))
    assert abs(O.reconstruction_error(t, V) - want) < 1e-12


def test_forward_by_scalar_loops():
    """y[b, l, o] = sum_c x[b, l, c] w[o, c], checked element by element."""
    rng = _rng(16)
    B, L, Cx, Cy = 2, 5, 7, 3
    x = rng.standard_normal((B, L, Cx))
    w = rng.standard_normal((Cy, Cx))
    y = O.forward(x, w)
    assert y.shape == (B, L, Cy)
    for b in range(B):
        for l in range(L):
            for o in range(Cy):
                acc = 0.0
                for c in range(Cx):
                    acc += x[b, l, c] * w[o, c]
                assert abs(y[b, l, o] - acc) < 1e-12
    # w = I gives x back; a permutation matrix permutes the channels
    assert np.array_equal(O.forward(x, np.eye(Cx)), x)
    perm = np.eye(Cx)[[3, 0, 6, 1, 5, 2, 4]]
    assert np.array_equal(O.forward(x, perm), x[:, :, [3, 0, 6, 1, 5, 2, 4]])


def test_forward_compress_returns_both_products():
    rng = _rng(17)
    B, L, Cx, Cy, Rx = 2, 16, 8, 6, 3
    x = rng.standard_normal((B, L, Cx))
    w = rng.standard_normal((Cy, Cx))
    P = _orthonormal_rows(rng, Rx, L)
    out = O.forward_compress(x, w, P)
    assert np.allclose(out["y"], O.forward(x, w), rtol=0, atol=0)
    assert np.allclose(out["x_hat"], O.compress_act(x, P), rtol=0, atol=0)
    # x_hat = P x: with P the first Rx unit rows, x_hat is the first Rx tokens
    E = np.eye(L)[:Rx]
    assert np.array_equal(O.forward_compress(x, w, E)["x_hat"], x[:, :Rx, :])
    # the forward FLOPs of one sample: 2 L Cx Cy (half the vanilla backward's 4 L Cx Cy)
    t = O.FlopTally()
    O.forward(x[:1], w, t)
    assert t.flops == 2 * L * Cx * Cy == O.flops_vanilla(L, Cx, Cy) // 2
