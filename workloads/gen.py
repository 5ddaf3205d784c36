"""Seeded generators for the synthetic workloads of the low-rank linear backward.

The workloads imitate the shapes and spectra of the INSTANT notes' experiments
(page "INSTANT: Compressing Gradients and Activations for Resource-Efficient
Training", sections 研究背景 / 关键设计 1-3 / 实验): a BERT-base block, a
transformer FFN pair, the EfficientFormer-L1 last stage (49 tokens) and a long,
wide linear.  No dataset is read: every tensor is drawn from numpy's PCG64 with
a documented seed.

Recipe (all readings of the workload descriptions):

* planted activations / gradients: ``t_b = U diag(sigma) V_b + noise``; ``U`` is
  the Q factor of a seeded Gaussian ``[L, m]`` shared by all samples of one
  tensor kind, ``V_b`` is per sample (orthonormal rows from a QR when
  ``orth_v``; otherwise ``Gaussian[m, C] / sqrt(C)`` so that ``E[V V^T] = I``).
* ``sigma_i = sigma_0 * i**(-alpha)``; with ``unit_rms`` the scale ``sigma_0`` is
  chosen so that the signal has unit RMS, ``sum sigma_i^2 = L * C``.
* noise ``N(0, var)``; the second argument of ``N(.,.)`` is read as a variance.
* bf16 tensors are rounded once, round-to-nearest-even, from the fp32 value;
  both the oracle and the CUDA path consume the same 16-bit patterns.

Seeds: ``0xC0FFEE + 1000 * seed_id + 500 * layer + tensor_id`` (each workload
has its own ``seed_id``) with tensor ids
x=1, g_y=2, w=3, calibration batch j: x=4+2j, g_y=5+2j; planted bases
U_x=400, U_g=401; drift planes 402.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED_BASE = 0xC0FFEE

TID_X, TID_G, TID_W = 1, 2, 3
TID_UX, TID_UG, TID_DRIFT = 400, 401, 402


def seed_for(seed_id: int, tensor_id: int, layer: int = 0) -> int:
    return SEED_BASE + 1000 * seed_id + 500 * layer + tensor_id


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# --------------------------------------------------------------------------
# bf16 encoding (round to nearest even) -- a storage format, not arithmetic
# of the method.
# --------------------------------------------------------------------------
def f32_to_bf16_bits(a) -> np.ndarray:
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# primitive generators
# --------------------------------------------------------------------------
def planted_basis(seed: int, L: int, m: int) -> np.ndarray:
    """Orthonormal ``[L, m]`` basis: Q factor of a seeded Gaussian."""
    g = _rng(seed).standard_normal((L, m))
    q, r = np.linalg.qr(g)
    # fix the QR sign freedom so the basis is a function of the seed alone
    q = q * np.sign(np.where(np.diag(r) == 0, 1.0, np.diag(r)))[None, :]
    return q


def sigma_profile(kind: str, m: int, L: int, C: int, unit_rms: bool,
                  alpha: float = 1.0) -> np.ndarray:
    """Planted singular values of one sample (length ``m``)."""
    i = np.arange(1, m + 1, dtype=np.float64)
    if kind == "pow2":
        s = 2.0 ** (-i)
    elif kind == "power":
        s = i ** (-alpha)
    else:
        raise ValueError(kind)
    if unit_rms:
        s = s * math.sqrt(L * C / float(np.sum(s * s)))
    return s


def planted_batch(seed: int, U: np.ndarray, sigma: np.ndarray, B: int, C: int,
                  noise_std: float, orth_v: bool, dtype=np.float64) -> np.ndarray:
    """``[B, L, C]`` samples ``U diag(sigma) V_b + noise_std * N(0, 1)``.

    Draw order from the seeded stream: all ``V_b`` (sample-major), then all
    noise (sample-major).  ``dtype`` is the precision the product is formed in.
    """
    L, m = U.shape
    rng = _rng(seed)
    US = (U * sigma[None, :]).astype(dtype)
    if orth_v:
        V = np.empty((B, m, C), dtype=dtype)
        for b in range(B):
            q, r = np.linalg.qr(rng.standard_normal((C, m)))
            q = q * np.sign(np.where(np.diag(r) == 0, 1.0, np.diag(r)))[None, :]
            V[b] = q.T
    else:
        V = rng.standard_normal((B, m, C), dtype=dtype)
        V *= dtype(1.0 / math.sqrt(C))
    t = np.matmul(US[None, :, :], V)
    if noise_std > 0:
        t += dtype(noise_std) * rng.standard_normal((B, L, C), dtype=dtype)
    return t.astype(np.float32)


def weight(seed: int, Cy: int, Cx: int, var: float) -> np.ndarray:
    return (_rng(seed).standard_normal((Cy, Cx)) * math.sqrt(var)).astype(np.float32)


def gelu_activations(seed: int, B: int, L: int, C: int) -> np.ndarray:
    """GELU (exact erf form, evaluated in fp64) of ``N(0, 1)`` pre-activations."""
    from scipy.special import erf

    z = _rng(seed).standard_normal((B, L, C))
    return (0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))).astype(np.float32)


def givens_rotate(U: np.ndarray, seed: int, step: int, angle: float) -> np.ndarray:
    """Rotate the token-space basis ``U [L, m]`` in one seeded plane ``(i, j)``."""
    L = U.shape[0]
    rng = _rng(seed + 7919 * step)
    i = int(rng.integers(0, L))
    j = int(rng.integers(0, L - 1))
    if j >= i:
        j += 1
    c, s = math.cos(angle), math.sin(angle)
    V = U.copy()
    ui, uj = U[i].copy(), U[j].copy()
    V[i] = c * ui - s * uj
    V[j] = s * ui + c * uj
    return V


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Workload:
    seed_id: int               # enters every seed of the workload's tensors
    name: str
    dtype: str                 # "f32" or "bf16"
    B: int
    L: int
    layers: tuple              # ((Cx, Cy), ...)
    Rx: int
    Ry: int
    x_kind: str                # "planted" | "gelu"
    x_sigma: str               # "pow2" | "power"
    x_alpha: float
    g_sigma: str
    g_alpha: float
    m_x: int                   # planted modes of x
    m_g: int                   # planted modes of g_y
    unit_rms: bool
    orth_v: bool
    noise_std: float
    w_var: float               # None -> 1/Cx
    calib_samples: int
    p: int
    eps: float = 0.95
    n_t: int = 100
    steps: int = 1
    drift_angle: float = 0.0

    @property
    def storage(self):
        return np.float32 if self.dtype == "f32" else np.uint16

    def w_variance(self, Cx: int) -> float:
        return (1.0 / Cx) if self.w_var is None else self.w_var


WORKLOADS = {
    "fp32_linear_64": Workload(1, "fp32 single linear 64x64", "f32", B=1, L=64, layers=((64, 64),),
                Rx=4, Ry=4, x_kind="planted", x_sigma="pow2", x_alpha=0.0,
                g_sigma="pow2", g_alpha=0.0, m_x=6, m_g=6, unit_rms=False,
                orth_v=True, noise_std=1e-3, w_var=None, calib_samples=8, p=2),
    "bert_base_block": Workload(2, "BERT-base block linear 768x768", "bf16", B=32, L=512,
                layers=((768, 768),), Rx=8, Ry=8, x_kind="planted", x_sigma="power",
                x_alpha=1.5, g_sigma="power", g_alpha=1.5, m_x=512, m_g=512,
                unit_rms=True, orth_v=False, noise_std=0.1, w_var=0.02,
                calib_samples=64, p=2),
    "bert_ffn_pair": Workload(3, "transformer FFN pair 768-3072-768", "bf16", B=32, L=512,
                layers=((768, 3072), (3072, 768)), Rx=16, Ry=16, x_kind="planted",
                x_sigma="power", x_alpha=1.2, g_sigma="power", g_alpha=1.2,
                m_x=512, m_g=512, unit_rms=True, orth_v=False, noise_std=0.1,
                w_var=0.02, calib_samples=64, p=2),
    "vit_mlp_pair_49": Workload(4, "ViT last-stage MLP pair 448-1792-448, 49 tokens", "bf16", B=256,
                L=49, layers=((448, 1792), (1792, 448)), Rx=8, Ry=8, x_kind="gelu",
                x_sigma="power", x_alpha=0.0, g_sigma="pow2", g_alpha=0.0, m_x=0,
                m_g=6, unit_rms=True, orth_v=False, noise_std=0.1, w_var=0.02,
                calib_samples=256, p=2, n_t=100, steps=20, drift_angle=0.05),
    "long_seq_4096_11008": Workload(5, "long-sequence wide linear 4096->11008, L=2048", "bf16", B=4,
                L=2048, layers=((4096, 11008),), Rx=16, Ry=16, x_kind="planted",
                x_sigma="power", x_alpha=1.0, g_sigma="power", g_alpha=1.0,
                m_x=512, m_g=512, unit_rms=True, orth_v=False, noise_std=0.1,
                w_var=0.02, calib_samples=64, p=4),
}


def workload(name: str, **overrides) -> Workload:
    """A workload by name: fp32_linear_64 (fp32, B=1, L=64, 64x64, R=4),
    bert_base_block (B=32, L=512, 768x768, R=8), bert_ffn_pair (768-3072-768,
    R=16), vit_mlp_pair_49 (B=256, L=49, 448-1792-448, R=8, drifting g_y) and
    long_seq_4096_11008 (B=4, L=2048, 4096->11008, R=16)."""
    wl = WORKLOADS[name]
    return dataclasses.replace(wl, **overrides) if overrides else wl


def _store(wl: Workload, a: np.ndarray) -> np.ndarray:
    return a.astype(np.float32) if wl.dtype == "f32" else f32_to_bf16_bits(a)


def _gen_dtype(wl: Workload):
    # fp32 workloads are formed in fp64 and stored in fp32; bf16 workloads are
    # formed in fp32 and rounded once to bf16.
    return np.float64 if wl.dtype == "f32" else np.float32


class LayerInputs:
    """Generator of one layer's stored tensors for a workload.

    Tensors come back in their stored form: ``float32`` arrays for fp32
    workloads, ``uint16`` bf16 bit patterns otherwise.
    """

    def __init__(self, wl: Workload, layer: int = 0, B: int | None = None):
        self.wl = wl
        self.layer = layer
        self.B = wl.B if B is None else B
        self.Cx, self.Cy = wl.layers[layer]
        L = wl.L
        self.Ux = None
        if wl.x_kind == "planted":
            self.Ux = planted_basis(seed_for(wl.seed_id, TID_UX, layer), L, wl.m_x)
            self.sx = sigma_profile(wl.x_sigma, wl.m_x, L, self.Cx, wl.unit_rms, wl.x_alpha)
        self.Ug = planted_basis(seed_for(wl.seed_id, TID_UG, layer), L, wl.m_g)
        self.sg = sigma_profile(wl.g_sigma, wl.m_g, L, self.Cy, wl.unit_rms, wl.g_alpha)

    def _x(self, seed: int, B: int) -> np.ndarray:
        wl = self.wl
        if wl.x_kind == "gelu":
            return gelu_activations(seed, B, wl.L, self.Cx)
        dt = _gen_dtype(wl)
        return planted_batch(seed, self.Ux, self.sx, B, self.Cx, wl.noise_std, wl.orth_v, dt)

    def _g(self, seed: int, B: int, step: int = 0) -> np.ndarray:
        wl = self.wl
        U = self.Ug
        if wl.drift_angle and step:
            for t in range(1, step + 1):
                U = givens_rotate(U, seed_for(wl.seed_id, TID_DRIFT, self.layer), t,
                                  wl.drift_angle)
        dt = _gen_dtype(wl)
        return planted_batch(seed, U, self.sg, B, self.Cy, wl.noise_std, wl.orth_v, dt)

    def x(self) -> np.ndarray:
        return _store(self.wl, self._x(seed_for(self.wl.seed_id, TID_X, self.layer), self.B))

    def g_y(self, step: int = 0) -> np.ndarray:
        s = seed_for(self.wl.seed_id, TID_G, self.layer) + 100_000 * step
        return _store(self.wl, self._g(s, self.B, step))

    def w(self) -> np.ndarray:
        wl = self.wl
        return _store(wl, weight(seed_for(wl.seed_id, TID_W, self.layer), self.Cy, self.Cx,
                                 wl.w_variance(self.Cx)))

    def calib_x(self, j: int, B: int) -> np.ndarray:
        return _store(self.wl, self._x(seed_for(self.wl.seed_id, 4 + 2 * j, self.layer), B))

    def calib_g(self, j: int, B: int, step: int = 0) -> np.ndarray:
        s = seed_for(self.wl.seed_id, 5 + 2 * j, self.layer) + 100_000 * step
        return _store(self.wl, self._g(s, B, step))
