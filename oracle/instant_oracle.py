"""fp64 CPU oracle of INSTANT low-rank backpropagation for one linear layer.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the GPU library computes.  It is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``; the
product path never imports it, and it imports nothing from the product path.

Source: the page "INSTANT: Compressing Gradients and Activations for
Resource-Efficient Training" (ICLR 2026 paper notes).  Section names below are
that page's:

* 整体框架 (overall framework): the forward ``y = x w^T`` is unchanged and the
  compressed activation ``x_hat = P x`` is stored instead of ``x``; ``P`` and
  ``Q`` are recalibrated every ``N_t`` steps.
* 关键设计 1: ``C_X = E[x x^T] = U Sigma U^T`` and ``C_G = E[g_y g_y^T]``; the
  left singular vectors give the projection; only the autocorrelation
  statistics are accumulated during calibration, the batch is not folded into
  the decomposition.
* 关键设计 2: ``E = sum_i sigma_i^2 = ||C_G||_F^2``; ``k`` is the smallest index
  with ``sum_{i<=k} sigma_i^2 >= eps * E``; rank ``k + p`` (oversampling);
  ``Q = U_{k+p}^T * (sum_{i<=k+p} sigma_i^2)^(-1/2)``, ``Q`` is ``[R_y, L]``; ``P``
  is formed the same way from ``C_X``; ``eps`` is fixed at 0.95.
* 关键设计 3: vanilla ``g_w = g_y^T x``, ``g_x = g_y w`` cost ``4 L C_x C_y``;
  low rank ``g_w ~ (g_y^T P^T)(P x) = g_hat_y1 x_hat``, ``g_hat_y2 = Q g_y``,
  ``g_hat_x = g_hat_y2 w``, ``g_tilde_x = Q^T g_hat_x``; cost
  ``2 (R_x + R_y)(C_x C_y + L C_x + L C_y)``; about 27x fewer FLOPs at
  ``L = 512, C_x = C_y = 768, R_x = R_y = 8``.

Readings taken where the page leaves a step open (each also listed in the
design notes):

1. ``sigma_i`` in the truncation rule and in the scale are the diagonal of
   ``Sigma`` in ``C = U Sigma U^T`` (eigenvalues of the symmetric PSD ``C``),
   since the page equates ``sum sigma_i^2`` with ``||C_G||_F^2``.
2. ``E[.]`` is the mean over the ``n`` accumulated samples.
3. The scale multiplies the whole ``[R, L]`` projector, exactly as written.
4. ``k >= 1``; ties at ``eps * E`` count as reached; ``R = min(k + p, L)``
   unless a rank is imposed.
5. Each eigenvector's sign is fixed so that its largest-magnitude entry is
   positive (lowest index on ties).

Precision: every input is decoded exactly as stored (bf16 bit patterns or fp32)
to fp64 and all arithmetic runs in fp64.  numpy's ``@`` (a matmul) and
``numpy.linalg.eigh`` (a symmetric eigendecomposition) are the only library
primitives used as steps.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "decode",
    "FlopTally",
    "compress_act",
    "project_grad",
    "grad_w",
    "grad_x_core",
    "expand",
    "grad_x",
    "low_rank_backward",
    "vanilla_backward",
    "forward",
    "forward_compress",
    "accumulate_autocorrelation",
    "eig_desc",
    "frobenius_energy",
    "truncation_index",
    "energy_scale",
    "canonical_sign",
    "calibrate",
    "flops_vanilla",
    "flops_low_rank",
    "reconstruction_error",
]


# ---------------------------------------------------------------------------
# storage decoding
# ---------------------------------------------------------------------------
def decode(a) -> np.ndarray:
    """Stored tensor -> fp64.  ``uint16`` arrays are bf16 bit patterns."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


class FlopTally:
    """Counts the floating-point work of every product the oracle performs.

    A product of an ``[a, b]`` by a ``[b, c]`` matrix is ``a*b*c`` multiply-adds,
    i.e. ``2*a*b*c`` flops -- the unit the page's closed forms use.
    """

    def __init__(self):
        self.flops = 0

    def mm(self, A: np.ndarray, Bm: np.ndarray) -> np.ndarray:
        a, b = A.shape[-2], A.shape[-1]
        c = Bm.shape[-1]
        batch = int(np.prod(np.broadcast_shapes(A.shape[:-2], Bm.shape[:-2]))) \
            if (A.ndim > 2 or Bm.ndim > 2) else 1
        self.flops += 2 * a * b * c * batch
        return A @ Bm


def _mm(tally, A, Bm):
    return tally.mm(A, Bm) if tally is not None else A @ Bm


# ---------------------------------------------------------------------------
# the per-step path (整体框架, 关键设计 3)
# ---------------------------------------------------------------------------
def compress_act(x, P, tally=None) -> np.ndarray:
    """Stored activation ``x_hat_b = P x_b``: ``[B,L,Cx], [Rx,L] -> [B,Rx,Cx]``."""
    x, P = decode(x), decode(P)
    return _mm(tally, P[None, :, :], x)


def project_grad(g_y, P, Q, tally=None):
    """``S_x,b = P g_y,b`` and ``S_q,b = Q g_y,b`` (``g_hat_y1,b = S_x,b^T``,
    ``g_hat_y2,b = S_q,b``): ``[B,L,Cy] -> [B,Rx,Cy], [B,Ry,Cy]``."""
    g, P, Q = decode(g_y), decode(P), decode(Q)
    return _mm(tally, P[None], g), _mm(tally, Q[None], g)


def grad_w(Sx, x_hat, tally=None) -> np.ndarray:
    """``g_w = sum_b g_hat_y1,b x_hat_b = sum_b S_x,b^T x_hat_b``: ``[Cy, Cx]``."""
    Sx, xh = np.asarray(Sx, np.float64), np.asarray(x_hat, np.float64)
    B = Sx.shape[0]
    gw = np.zeros((Sx.shape[2], xh.shape[2]))
    for b in range(B):
        gw += _mm(tally, Sx[b].T, xh[b])
    return gw


def grad_x_core(Sq, w, tally=None) -> np.ndarray:
    """``g_hat_x,b = g_hat_y2,b w``: ``[B,Ry,Cy], [Cy,Cx] -> [B,Ry,Cx]``."""
    return _mm(tally, np.asarray(Sq, np.float64), decode(w)[None])


def expand(Q, gx_hat, tally=None) -> np.ndarray:
    """``g_tilde_x,b = Q^T g_hat_x,b``: ``[Ry,L], [B,Ry,Cx] -> [B,L,Cx]``."""
    Q = decode(Q)
    return _mm(tally, Q.T[None], np.asarray(gx_hat, np.float64))


def grad_x(Sq, w, Q, tally=None) -> np.ndarray:
    """``g_tilde_x = Q^T (S_q w)`` per sample."""
    return expand(Q, grad_x_core(Sq, w, tally), tally)


def low_rank_backward(x, g_y, w, P, Q, tally=None) -> dict:
    """One layer's compress + low-rank backward, every intermediate returned."""
    xh = compress_act(x, P, tally)
    Sx, Sq = project_grad(g_y, P, Q, tally)
    gw = grad_w(Sx, xh, tally)
    gxh = grad_x_core(Sq, w, tally)
    gx = expand(Q, gxh, tally)
    return {"x_hat": xh, "Sx": Sx, "Sq": Sq, "g_w": gw, "gx_hat": gxh, "g_x": gx}


def forward(x, w, tally=None) -> np.ndarray:
    """The layer's forward ``y_b = x_b w^T``: ``[B,L,Cx], [Cy,Cx] -> [B,L,Cy]``
    (整体框架: the forward product itself is left as it is)."""
    x, w = decode(x), decode(w)
    return _mm(tally, x, w.T[None])


def forward_compress(x, w, P, tally=None) -> dict:
    """The forward pass as INSTANT runs it: ``y = x w^T`` and the stored
    activation ``x_hat = P x`` (整体框架: x_hat is kept instead of x)."""
    return {"y": forward(x, w, tally), "x_hat": compress_act(x, P, tally)}


def vanilla_backward(x, g_y, w, tally=None) -> dict:
    """Full-rank ``g_w = sum_b g_y,b^T x_b`` and ``g_x,b = g_y,b w``."""
    x, g, w = decode(x), decode(g_y), decode(w)
    gw = np.zeros((g.shape[2], x.shape[2]))
    for b in range(x.shape[0]):
        gw += _mm(tally, g[b].T, x[b])
    gx = _mm(tally, g, w[None])
    return {"g_w": gw, "g_x": gx}


# ---------------------------------------------------------------------------
# calibration (关键设计 1 and 2)
# ---------------------------------------------------------------------------
def accumulate_autocorrelation(t, C_sum=None) -> np.ndarray:
    """Unnormalised statistic ``C_sum + sum_b t_b t_b^T`` (``L x L``).

    Dividing by the number of accumulated samples gives ``E[t t^T]``."""
    t = decode(t)
    L = t.shape[1]
    out = np.zeros((L, L)) if C_sum is None else np.array(C_sum, np.float64, copy=True)
    for b in range(t.shape[0]):
        out += t[b] @ t[b].T
    return out


def eig_desc(C):
    """Eigenpairs of the symmetric ``C``, eigenvalues in descending order."""
    C = np.asarray(C, np.float64)
    lam, U = np.linalg.eigh(0.5 * (C + C.T))
    order = np.argsort(lam)[::-1]
    return lam[order], U[:, order]


def frobenius_energy(C) -> float:
    """``E = ||C||_F^2 = sum_ij C_ij^2``."""
    C = np.asarray(C, np.float64)
    return float(np.sum(C * C))


def truncation_index(lam_desc, E: float, eps: float) -> int:
    """Smallest ``k >= 1`` with ``sum_{i<=k} sigma_i^2 >= eps * E``.

    Returns ``len(lam_desc) + 1`` when the listed values never reach it."""
    target = eps * E
    acc = 0.0
    for i, s in enumerate(np.asarray(lam_desc, np.float64)):
        acc += s * s
        if acc >= target:
            return i + 1
    return len(lam_desc) + 1


def energy_scale(lam_desc, R: int) -> float:
    """``(sum_{i<=R} sigma_i^2)^(-1/2)``."""
    lam = np.asarray(lam_desc, np.float64)[:R]
    return float(1.0 / np.sqrt(np.sum(lam * lam)))


def canonical_sign(U) -> np.ndarray:
    """Flip each column so that its largest-magnitude entry is positive."""
    U = np.array(U, np.float64, copy=True)
    for j in range(U.shape[1]):
        i = int(np.argmax(np.abs(U[:, j])))
        if U[i, j] < 0:
            U[:, j] = -U[:, j]
    return U


def calibrate(C_sum, n_samples: int, eps: float = 0.95, p: int = 0,
              r_override: int = 0, scale_on: bool = True) -> dict:
    """Projector rows from an accumulated autocorrelation.

    ``C = C_sum / n``; ``C = U Sigma U^T``; ``E = ||C||_F^2``; ``k`` by the
    energy rule; ``R = min(k + p, L)`` (or ``r_override``); rows
    ``s * U_R^T`` with ``s = (sum_{i<=R} sigma_i^2)^(-1/2)`` (1 when the scale
    is off)."""
    C = np.asarray(C_sum, np.float64) / float(n_samples)
    L = C.shape[0]
    E = frobenius_energy(C)
    if not np.isfinite(E) or E <= 0.0:
        raise FloatingPointError("autocorrelation has no finite positive energy")
    lam, U = eig_desc(C)
    k = min(truncation_index(lam, E, eps), L)
    R = r_override if r_override > 0 else min(k + p, L)
    s = energy_scale(lam, R) if scale_on else 1.0
    Ur = canonical_sign(U[:, :R])
    return {"k": k, "R": R, "scale": s, "rows": s * Ur.T, "eigenvalues": lam,
            "energy": E, "C": C}


# ---------------------------------------------------------------------------
# closed forms and diagnostics
# ---------------------------------------------------------------------------
def flops_vanilla(L: int, Cx: int, Cy: int) -> int:
    """Vanilla backward of one linear layer: ``4 L Cx Cy`` (关键设计 3)."""
    return 4 * L * Cx * Cy


def flops_low_rank(L: int, Cx: int, Cy: int, Rx: int, Ry: int) -> int:
    """Low-rank compress + backward: ``2 (Rx + Ry)(Cx Cy + L Cx + L Cy)``."""
    return 2 * (Rx + Ry) * (Cx * Cy + L * Cx + L * Cy)


def reconstruction_error(t, rows) -> float:
    """``||t - V^T V t||_F / ||t||_F`` for orthonormal projector rows ``V``."""
    t = decode(t)
    V = np.asarray(rows, np.float64)
    rec = V.T[None] @ (V[None] @ t)
    return float(np.linalg.norm(t - rec) / np.linalg.norm(t))
