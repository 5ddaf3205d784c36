"""Per-layer driver of INSTANT low-rank backpropagation for ``y = x w^T``.

Holds the state the method keeps for one linear layer -- the stacked projector
``[P; Q]``, the calibration statistics and the step counter -- plus the
preallocated device buffers, and sequences the library calls of one training
step (page "INSTANT: Compressing Gradients and Activations for
Resource-Efficient Training", 整体框架: P and Q are recalibrated every N_t
steps; the forward stores x_hat = P x; the backward uses low-rank products).
Every arithmetic step runs in the CUDA library; torch only owns memory.
"""

from __future__ import annotations

import torch

from . import api


class InstantLinear:
    def __init__(self, w: torch.Tensor, B: int, L: int, Rx: int, Ry: int, *, n_t: int = 100,
                 eps: float = 0.95, p: int = 2, scale_on: bool = True):
        if w.dim() != 2 or not w.is_cuda:
            raise ValueError("w must be a [Cy, Cx] CUDA tensor")
        self.w = w
        self.dtype = w.dtype
        self.Cy, self.Cx = w.shape
        self.B, self.L, self.Rx, self.Ry = B, L, Rx, Ry
        self.n_t, self.eps, self.p, self.scale_on = n_t, eps, p, scale_on
        dev = w.device
        f32 = torch.float32
        self.PQ = torch.zeros(Rx + Ry, L, dtype=self.dtype, device=dev)
        self.C_X = torch.zeros(L, L, dtype=f32, device=dev)
        self.C_G = torch.zeros(L, L, dtype=f32, device=dev)
        self.n_x = 0
        self.n_g = 0
        self.t = 0
        self.xhat = torch.empty(B, Rx, self.Cx, dtype=self.dtype, device=dev)
        self.Sx = torch.empty(B * Rx, self.Cy, dtype=self.dtype, device=dev)
        self.Sq = torch.empty(B * Ry, self.Cy, dtype=self.dtype, device=dev)
        self.gw = torch.empty(self.Cy, self.Cx, dtype=f32, device=dev)
        self.gx = torch.empty(B, L, self.Cx, dtype=self.dtype, device=dev)
        nbytes = api.grad_x_workspace_bytes(B, L, self.Cx, self.Cy, Ry, self.dtype)
        self.ws_gx = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
        self.ws_bw = api.backward_workspace(B, L, self.Cx, self.Cy, Ry, self.dtype, dev)
        self.ws_cal = torch.empty(api.calib_batch_workspace_bytes(L, 2), dtype=torch.uint8,
                                  device=dev)
        self.last_calibration = None
        self._cal = None   # the solve's argument block, built on first use
        self.ws_fwd = None  # forward workspace (zeroed), built on first use

    # views of the stacked projector
    @property
    def P(self) -> torch.Tensor:
        return self.PQ[: self.Rx]

    @property
    def Q(self) -> torch.Tensor:
        return self.PQ[self.Rx:]

    # ---- the per-step path -------------------------------------------------
    def forward(self, x: torch.Tensor, y: torch.Tensor | None = None,
                xhat: torch.Tensor | None = None) -> torch.Tensor:
        """The layer's forward ``y = x w^T``; the compressed activation
        ``x_hat = P x`` is formed from the same pass over ``x`` and kept for the
        backward (returns ``y``)."""
        B, L, _ = x.shape
        if y is None:
            y = torch.empty(B, L, self.Cy, dtype=self.dtype, device=x.device)
        if self.ws_fwd is None:
            self.ws_fwd = api.forward_workspace(self.B, self.L, self.Cx, self.Rx, self.dtype,
                                                x.device)
        api.forward(x, self.w, y, self.P, self.xhat if xhat is None else xhat, self.ws_fwd)
        return y

    def compress(self, x: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
        """Forward-side activation compression ``x_hat = P x``."""
        return api.compress_act(x, self.P, self.xhat if out is None else out)

    def backward(self, g_y: torch.Tensor, xhat: torch.Tensor | None = None,
                 gw: torch.Tensor | None = None, gx: torch.Tensor | None = None,
                 accumulate: bool = False):
        """Low-rank backward: returns ``(g_w, g_tilde_x)``."""
        xhat = self.xhat if xhat is None else xhat
        gw = self.gw if gw is None else gw
        gx = self.gx if gx is None else gx
        api.backward(g_y, self.PQ, xhat, self.w, self.Sx, self.Sq, gw, gx, self.ws_bw, self.Rx,
                     accumulate=accumulate)
        return gw, gx

    # ---- calibration --------------------------------------------------------
    def accumulate(self, x: torch.Tensor | None = None, g_y: torch.Tensor | None = None) -> None:
        """Adds the autocorrelation statistics of a batch (no batch is stored)."""
        pairs = []
        if x is not None:
            pairs.append((x, self.C_X))
            self.n_x += x.shape[0]
        if g_y is not None:
            pairs.append((g_y, self.C_G))
            self.n_g += g_y.shape[0]
        if pairs:
            api.calib_accumulate_batch(pairs)   # both statistics in one launch

    def recalibrate(self, r_override: bool = True):
        """Solves both statistics into ``P`` and ``Q`` (one call) and clears them.

        With ``r_override`` the ranks stay at the buffer sizes ``Rx``/``Ry``;
        ``k`` and ``k + p`` are still reported."""
        if self.n_x == 0 or self.n_g == 0:
            raise RuntimeError("recalibrate: no statistics accumulated")
        warm = self.last_calibration is not None
        if self._cal is None:
            common = dict(eps=self.eps, p=self.p, scale_on=self.scale_on)
            self._cal = api.CalibBatch([dict(C=self.C_X, rows_out=self.P, **common),
                                        dict(C=self.C_G, rows_out=self.Q, **common)], self.ws_cal)
        rx, rg = self._cal.solve(
            (self.n_x, self.n_g), warm_start=warm,
            r_override=(self.Rx if r_override else 0, self.Ry if r_override else 0))
        self.C_X.zero_()
        self.C_G.zero_()
        self.n_x = self.n_g = 0
        self.last_calibration = (rx, rg)
        return rx, rg

    def step(self, x: torch.Tensor, g_y: torch.Tensor, calib=()):
        """One training step of the layer on the recalibration schedule.

        Every ``n_t`` steps the statistics of this batch (and of the extra
        calibration batches ``calib``, pairs ``(x_c, g_c)``) are accumulated
        and solved; then the activation is compressed and the low-rank
        backward runs."""
        if self.t % self.n_t == 0:
            self.accumulate(x, g_y)
            for xc, gc in calib:
                self.accumulate(xc, gc)
            self.recalibrate()
        self.compress(x)
        out = self.backward(g_y)
        self.t += 1
        return out


class LayerCalibration:
    """The recalibration of several layers at the same step (整体框架: every
    layer recalibrates every N_t steps, so a model's layers do it together):
    the statistics of all of them -- each layer's ``C_X`` into ``P`` and
    ``C_G`` into ``Q`` -- go to ``instant_calib_solve_batch`` in one call
    (one launch where the one-launch solver takes the token length, up to 16
    statistics), instead of one call per layer.  Each layer gets the results
    its own :meth:`InstantLinear.recalibrate` would give it (bit for bit where
    the one-launch cluster solver takes L, 128 < L <= 2048).  The layers must
    share the token length L and the dtype; the argument block and the
    workspace are built once."""

    def __init__(self, layers):
        self.layers = list(layers)
        if not self.layers:
            raise ValueError("LayerCalibration: no layers")
        L, dt = self.layers[0].L, self.layers[0].dtype
        if any(l.L != L or l.dtype != dt for l in self.layers):
            raise ValueError("LayerCalibration: layers differ in L or dtype")
        self.batches = []
        # at most 8 layers (16 statistics) per call
        for i in range(0, len(self.layers), 8):
            group = self.layers[i:i + 8]
            ws = torch.empty(api.calib_batch_workspace_bytes(L, 2 * len(group)), dtype=torch.uint8,
                             device=group[0].w.device)
            probs = []
            for l in group:
                common = dict(eps=l.eps, p=l.p, scale_on=l.scale_on)
                probs += [dict(C=l.C_X, rows_out=l.P, **common), dict(C=l.C_G, rows_out=l.Q, **common)]
            self.batches.append((group, api.CalibBatch(probs, ws), ws))

    def recalibrate(self, r_override: bool = True):
        """Solves every layer's statistics and clears them; returns the list of
        ``(result_x, result_g)`` per layer."""
        out = []
        for group, batch, _ in self.batches:
            if any(l.n_x == 0 or l.n_g == 0 for l in group):
                raise RuntimeError("recalibrate: no statistics accumulated")
            warm = all(l.last_calibration is not None for l in group)
            counts, over = [], []
            for l in group:
                counts += [l.n_x, l.n_g]
                over += [l.Rx if r_override else 0, l.Ry if r_override else 0]
            res = batch.solve(counts, warm_start=warm, r_override=over)
            for i, l in enumerate(group):
                l.C_X.zero_()
                l.C_G.zero_()
                l.n_x = l.n_g = 0
                l.last_calibration = (res[2 * i], res[2 * i + 1])
                out.append(l.last_calibration)
        return out
