"""Seeded input generators: determinism, shapes, spectra and bf16 rounding."""

import numpy as np
import pytest

import workloads as W


def test_bf16_rounding_matches_torch_rne():
    torch = pytest.importorskip("torch")
    rng = np.random.Generator(np.random.PCG64(1))
    f = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 10,
                        # exact halfway cases: low 16 bits 0x8000, both parities
                        (np.arange(64, dtype=np.uint32) << 16 | 0x3F800000 | 0x8000)
                        .view(np.float32)])
    ours = W.f32_to_bf16_bits(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = W.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16)
                          .to(torch.float32).numpy())


def test_generators_are_deterministic_and_shaped():
    wl = W.workload("fp32_linear_64")
    a = W.LayerInputs(wl)
    b = W.LayerInputs(wl)
    assert np.array_equal(a.x(), b.x())
    assert np.array_equal(a.g_y(), b.g_y())
    assert a.x().shape == (1, 64, 64) and a.x().dtype == np.float32
    assert a.w().shape == (64, 64)
    assert not np.array_equal(a.calib_x(0, 8), a.calib_x(1, 8))


def test_planted_spectrum_shape():
    # rank-6 pow2 spectrum plus 1e-3 noise; a 64x64 noise matrix has its top
    # singular value near 1e-3 * (8 + 8) = 0.016, comparable to sigma_6 = 2^-6
    wl = W.workload("fp32_linear_64")
    li = W.LayerInputs(wl)
    x = li.calib_x(0, 8).astype(np.float64)
    s = np.linalg.svd(x[0], compute_uv=False)
    assert np.allclose(s[:4], 2.0 ** -np.arange(1, 5), rtol=0.05)
    assert s[6] < 0.02


def test_givens_drift_keeps_orthonormality():
    U = W.planted_basis(5, 20, 4)
    V = W.givens_rotate(U, 9, 1, 0.05)
    assert np.allclose(V.T @ V, np.eye(4), atol=1e-12)
    assert not np.allclose(U, V)
