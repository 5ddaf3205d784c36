"""Python binding of the C ABI, one function per entry point of include/instant.h.

Each function takes torch CUDA tensors, checks their shapes against each other,
and passes raw device pointers, extents and the current CUDA stream to the
library.  No arithmetic of the method happens here.
"""

from __future__ import annotations

import ctypes
import dataclasses

import torch

from ._lib import (GRAD_X_STATIC_SCRATCH_BYTES, INSTANT_BF16, INSTANT_F32, AccumulateItem,
                   CalibParams, CalibProblem, check, lib)

__all__ = [
    "compress_act",
    "forward",
    "forward_workspace",
    "project_grad",
    "grad_w",
    "grad_x",
    "grad_x_workspace_bytes",
    "grad_w_x",
    "backward",
    "backward_workspace",
    "backward_workspace_bytes",
    "grad_x_core",
    "expand",
    "grad_x_static",
    "launch_count",
    "calib_accumulate",
    "calib_accumulate_batch",
    "calib_solve",
    "calib_solve_batch",
    "CalibBatch",
    "calib_workspace_bytes",
    "calib_batch_workspace_bytes",
    "device_status",
    "reconstruction_error",
    "CalibResult",
    "dtype_code",
]


def dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return INSTANT_BF16
    if t == torch.float32:
        return INSTANT_F32
    raise TypeError(f"unsupported dtype {t}: use torch.bfloat16 or torch.float32")


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _same_dtype(dt, *pairs):
    for name, t in pairs:
        if t.dtype != dt:
            raise TypeError(f"{name} has dtype {t.dtype}, expected {dt}")


def compress_act(x: torch.Tensor, P: torch.Tensor, xhat: torch.Tensor, stream=None) -> torch.Tensor:
    """``xhat[b] = P @ x[b]``: x ``[B, L, Cx]``, P ``[Rx, L]``, xhat ``[B, Rx, Cx]``."""
    B, L, Cx = x.shape
    Rx = P.shape[0]
    if P.shape != (Rx, L) or xhat.shape != (B, Rx, Cx):
        raise ValueError("compress_act: inconsistent shapes")
    _same_dtype(x.dtype, ("P", P), ("xhat", xhat))
    check(lib().instant_compress_act(_dev(x, "x"), _dev(P, "P"), _dev(xhat, "xhat"), B, L, Cx, Rx,
                                     dtype_code(x.dtype), _stream(stream)), "instant_compress_act")
    return xhat


def forward_workspace(B: int, L: int, Cx: int, Rx: int, dtype: torch.dtype, device) -> torch.Tensor:
    """A zeroed workspace for :func:`forward` (it must start at zero; every call
    leaves it zero)."""
    n = int(lib().instant_forward_workspace_bytes(B, L, Cx, Rx, dtype_code(dtype)))
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def forward(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, P: torch.Tensor | None = None,
            xhat: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    """``y[b] = x[b] w^T`` and, with ``P``, ``xhat[b] = P x[b]`` in the same pass:
    x ``[B, L, Cx]``, w ``[Cy, Cx]``, y ``[B, L, Cy]``, P ``[Rx, L]``,
    xhat ``[B, Rx, Cx]``; ws from :func:`forward_workspace`."""
    B, L, Cx = x.shape
    Cy = w.shape[0]
    if w.shape != (Cy, Cx) or y.shape != (B, L, Cy):
        raise ValueError("forward: inconsistent shapes")
    Rx = 0
    if P is not None:
        Rx = P.shape[0]
        if P.shape != (Rx, L) or xhat is None or xhat.shape != (B, Rx, Cx) or ws is None:
            raise ValueError("forward: P needs xhat [B, Rx, Cx] and a workspace")
        _same_dtype(x.dtype, ("P", P), ("xhat", xhat))
    _same_dtype(x.dtype, ("w", w), ("y", y))
    check(lib().instant_forward(_dev(x, "x"), _dev(w, "w"), _dev(P, "P") if P is not None else None,
                                _dev(y, "y"), _dev(xhat, "xhat") if P is not None else None,
                                _dev(ws, "ws") if ws is not None else None,
                                ws.numel() * ws.element_size() if ws is not None else 0, B, L, Cx,
                                Cy, Rx, dtype_code(x.dtype), _stream(stream)), "instant_forward")
    return y, xhat


def project_grad(g_y: torch.Tensor, PQ: torch.Tensor, Sx: torch.Tensor, Sq: torch.Tensor,
                 Rx: int, Ry: int, stream=None):
    """``Sx[b] = P g_y[b]``, ``Sq[b] = Q g_y[b]`` with ``PQ = [P; Q]``.

    g_y ``[B, L, Cy]``, PQ ``[Rx+Ry, L]``, Sx ``[B*Rx, Cy]``, Sq ``[B*Ry, Cy]``."""
    B, L, Cy = g_y.shape
    if PQ.shape != (Rx + Ry, L) or Sx.shape != (B * Rx, Cy) or Sq.shape != (B * Ry, Cy):
        raise ValueError("project_grad: inconsistent shapes")
    _same_dtype(g_y.dtype, ("PQ", PQ), ("Sx", Sx), ("Sq", Sq))
    check(lib().instant_project_grad(_dev(g_y, "g_y"), _dev(PQ, "PQ"), _dev(Sx, "Sx"), _dev(Sq, "Sq"),
                                     B, L, Cy, Rx, Ry, dtype_code(g_y.dtype), _stream(stream)),
          "instant_project_grad")
    return Sx, Sq


def grad_w(Sx: torch.Tensor, xhat: torch.Tensor, gw: torch.Tensor, B: int, accumulate: bool = False,
           stream=None) -> torch.Tensor:
    """``gw (+)= Sx^T xhat``: Sx ``[B*Rx, Cy]``, xhat ``[B*Rx, Cx]`` (or ``[B, Rx, Cx]``),
    gw ``[Cy, Cx]`` fp32."""
    K, Cy = Sx.shape
    xh = xhat.reshape(K, -1) if xhat.dim() == 3 else xhat
    Cx = xh.shape[1]
    if K % B != 0 or xh.shape[0] != K or gw.shape != (Cy, Cx) or gw.dtype != torch.float32:
        raise ValueError("grad_w: inconsistent shapes")
    _same_dtype(Sx.dtype, ("xhat", xhat))
    check(lib().instant_grad_w(_dev(Sx, "Sx"), _dev(xhat, "xhat"), _dev(gw, "gw"), int(bool(accumulate)),
                               B, K // B, Cx, Cy, dtype_code(Sx.dtype), _stream(stream)),
          "instant_grad_w")
    return gw


def grad_x_workspace_bytes(B: int, L: int, Cx: int, Cy: int, Ry: int, dtype: torch.dtype) -> int:
    return int(lib().instant_grad_x_workspace_bytes(B, L, Cx, Cy, Ry, dtype_code(dtype)))


def grad_x(Sq: torch.Tensor, w: torch.Tensor, Q: torch.Tensor, gx: torch.Tensor,
           ws: torch.Tensor, stream=None) -> torch.Tensor:
    """``gx[b] = Q^T (Sq[b] w)``: Sq ``[B*Ry, Cy]``, w ``[Cy, Cx]``, Q ``[Ry, L]``,
    gx ``[B, L, Cx]``; ws is scratch of ``grad_x_workspace_bytes`` bytes."""
    B, L, Cx = gx.shape
    Ry = Q.shape[0]
    Cy = w.shape[0]
    if Q.shape != (Ry, L) or w.shape != (Cy, Cx) or Sq.shape != (B * Ry, Cy):
        raise ValueError("grad_x: inconsistent shapes")
    _same_dtype(Sq.dtype, ("w", w), ("Q", Q), ("gx", gx))
    check(lib().instant_grad_x(_dev(Sq, "Sq"), _dev(w, "w"), _dev(Q, "Q"), _dev(gx, "gx"),
                               _dev(ws, "ws"), ws.numel() * ws.element_size(), B, L, Cx, Cy, Ry,
                               dtype_code(Sq.dtype), _stream(stream)), "instant_grad_x")
    return gx


def grad_w_x(Sx: torch.Tensor, xhat: torch.Tensor, gw: torch.Tensor, Sq: torch.Tensor,
             w: torch.Tensor, Q: torch.Tensor, gx: torch.Tensor, ws: torch.Tensor, B: int, *,
             accumulate: bool = False, stream=None):
    """:func:`grad_w` and :func:`grad_x` in one call (one launch where the
    single-kernel input gradient applies).  Returns ``(gw, gx)``."""
    Bg, L, Cx = gx.shape
    Ry = Q.shape[0]
    Cy = w.shape[0]
    Rx = Sx.shape[0] // B
    if (Bg != B or Q.shape != (Ry, L) or w.shape != (Cy, Cx) or Sq.shape != (B * Ry, Cy)
            or Sx.shape != (B * Rx, Cy) or xhat.numel() != B * Rx * Cx or gw.shape != (Cy, Cx)):
        raise ValueError("grad_w_x: inconsistent shapes")
    if gw.dtype != torch.float32:
        raise TypeError("grad_w_x: gw must be float32")
    _same_dtype(Sq.dtype, ("Sx", Sx), ("xhat", xhat), ("w", w), ("Q", Q), ("gx", gx))
    check(lib().instant_grad_w_x(_dev(Sx, "Sx"), _dev(xhat, "xhat"), _dev(gw, "gw"), int(bool(accumulate)),
                                 _dev(Sq, "Sq"), _dev(w, "w"), _dev(Q, "Q"), _dev(gx, "gx"),
                                 _dev(ws, "ws"), ws.numel() * ws.element_size(), B, L, Cx, Cy, Rx,
                                 Ry, dtype_code(Sq.dtype), _stream(stream)), "instant_grad_w_x")
    return gw, gx


def backward_workspace_bytes(B: int, L: int, Cx: int, Cy: int, Ry: int, dtype: torch.dtype) -> int:
    return int(lib().instant_backward_workspace_bytes(B, L, Cx, Cy, Ry, dtype_code(dtype)))


def backward_workspace(B: int, L: int, Cx: int, Cy: int, Ry: int, dtype: torch.dtype,
                       device) -> torch.Tensor:
    """A zeroed workspace for :func:`backward` (its counters must start at zero)."""
    return torch.zeros(backward_workspace_bytes(B, L, Cx, Cy, Ry, dtype), dtype=torch.uint8,
                       device=device)


def backward(g_y: torch.Tensor, PQ: torch.Tensor, xhat: torch.Tensor, w: torch.Tensor,
             Sx: torch.Tensor, Sq: torch.Tensor, gw: torch.Tensor, gx: torch.Tensor,
             ws: torch.Tensor, Rx: int, *, accumulate: bool = False, stream=None):
    """:func:`project_grad` then :func:`grad_w_x` in one call (one launch where
    the single-kernel input gradient applies).  ``ws`` comes from
    :func:`backward_workspace`.  Returns ``(gw, gx)``."""
    B, L, Cy = g_y.shape
    Ry = PQ.shape[0] - Rx
    Cx = w.shape[1]
    if (PQ.shape[1] != L or Ry < 1 or w.shape != (Cy, Cx) or xhat.numel() != B * Rx * Cx
            or Sx.shape != (B * Rx, Cy) or Sq.shape != (B * Ry, Cy) or gw.shape != (Cy, Cx)
            or gx.shape != (B, L, Cx)):
        raise ValueError("backward: inconsistent shapes")
    if gw.dtype != torch.float32:
        raise TypeError("backward: gw must be float32")
    _same_dtype(g_y.dtype, ("PQ", PQ), ("xhat", xhat), ("w", w), ("Sx", Sx), ("Sq", Sq), ("gx", gx))
    check(lib().instant_backward(_dev(g_y, "g_y"), _dev(PQ, "PQ"), _dev(xhat, "xhat"), _dev(w, "w"),
                                 _dev(Sx, "Sx"), _dev(Sq, "Sq"), _dev(gw, "gw"),
                                 int(bool(accumulate)), _dev(gx, "gx"), _dev(ws, "ws"),
                                 ws.numel() * ws.element_size(), B, L, Cx, Cy, Rx, Ry,
                                 dtype_code(g_y.dtype), _stream(stream)), "instant_backward")
    return gw, gx


def grad_x_core(Sq: torch.Tensor, w: torch.Tensor, ws: torch.Tensor, B: int, stream=None):
    """First half of :func:`grad_x`: ``g_hat_x = Sq w`` into the workspace."""
    Cy, Cx = w.shape
    Ry = Sq.shape[0] // B
    if Sq.shape != (B * Ry, Cy):
        raise ValueError("grad_x_core: inconsistent shapes")
    _same_dtype(Sq.dtype, ("w", w))
    check(lib().instant_grad_x_core(_dev(Sq, "Sq"), _dev(w, "w"), _dev(ws, "ws"),
                                    ws.numel() * ws.element_size(), B, Cx, Cy, Ry,
                                    dtype_code(Sq.dtype), _stream(stream)), "instant_grad_x_core")
    return ws


def grad_x_static(Sq: torch.Tensor, w: torch.Tensor, Q: torch.Tensor, gx: torch.Tensor,
                  stream=None) -> torch.Tensor:
    """:func:`grad_x` for callers that cannot allocate device memory: no
    workspace argument; ``g_hat_x`` lives in a fixed array of the library
    (``GRAD_X_STATIC_SCRATCH_BYTES`` per device) that every call on a device
    shares, so calls must not overlap in time.  The first call on a device
    looks the array up and should come before any stream capture."""
    B, L, Cx = gx.shape
    Ry = Q.shape[0]
    Cy = w.shape[0]
    if Q.shape != (Ry, L) or w.shape != (Cy, Cx) or Sq.shape != (B * Ry, Cy):
        raise ValueError("grad_x_static: inconsistent shapes")
    _same_dtype(Sq.dtype, ("w", w), ("Q", Q), ("gx", gx))
    status = lib().instant_grad_x_static(_dev(Sq, "Sq"), _dev(w, "w"), _dev(Q, "Q"), _dev(gx, "gx"),
                                         B, L, Cx, Cy, Ry, dtype_code(Sq.dtype), _stream(stream))
    if status == 5:
        need = grad_x_workspace_bytes(B, L, Cx, Cy, Ry, Sq.dtype)
        raise ValueError(f"grad_x_static: g_hat_x needs {need} bytes, more than the "
                         f"{GRAD_X_STATIC_SCRATCH_BYTES}-byte fixed array; use grad_x with a workspace")
    check(status, "instant_grad_x_static")
    return gx


def expand(Q: torch.Tensor, gx: torch.Tensor, ws: torch.Tensor, Cy: int, stream=None):
    """Second half of :func:`grad_x`: ``gx[b] = Q^T g_hat_x[b]`` from the workspace."""
    B, L, Cx = gx.shape
    Ry = Q.shape[0]
    if Q.shape != (Ry, L):
        raise ValueError("expand: inconsistent shapes")
    _same_dtype(Q.dtype, ("gx", gx))
    check(lib().instant_expand(_dev(Q, "Q"), _dev(gx, "gx"), _dev(ws, "ws"),
                               ws.numel() * ws.element_size(), B, L, Cx, Cy, Ry,
                               dtype_code(Q.dtype), _stream(stream)), "instant_expand")
    return gx


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().instant_launch_count())


def calib_accumulate(t: torch.Tensor, C: torch.Tensor, stream=None) -> torch.Tensor:
    """``C += sum_b t[b] t[b]^T``: t ``[B, L, C]``, C ``[L, L]`` fp32."""
    B, L, Cd = t.shape
    if C.shape != (L, L) or C.dtype != torch.float32:
        raise ValueError("calib_accumulate: C must be [L, L] float32")
    check(lib().instant_calib_accumulate(_dev(t, "t"), _dev(C, "C"), B, L, Cd, dtype_code(t.dtype),
                                         _stream(stream)), "instant_calib_accumulate")
    return C


def calib_accumulate_batch(pairs, stream=None) -> None:
    """``C += sum_b t[b] t[b]^T`` for every ``(t, C)`` in ``pairs`` (one token
    length L; t ``[B, L, Cdim]`` of one dtype, C ``[L, L]`` fp32), up to four
    statistics per launch."""
    pairs = list(pairs)
    if not pairs:
        raise ValueError("calib_accumulate_batch: nothing to accumulate")
    L = pairs[0][0].shape[1]
    dt = pairs[0][0].dtype
    arr = (AccumulateItem * len(pairs))()
    for i, (t, C) in enumerate(pairs):
        B, Lt, Cd = t.shape
        if Lt != L or t.dtype != dt or C.shape != (L, L) or C.dtype != torch.float32:
            raise ValueError("calib_accumulate_batch: inconsistent shapes or dtypes")
        arr[i] = AccumulateItem(_dev(t, "t"), _dev(C, "C"), B, Cd)
    check(lib().instant_calib_accumulate_batch(arr, len(pairs), L, dtype_code(dt), _stream(stream)),
          "instant_calib_accumulate_batch")


def calib_workspace_bytes(L: int, r_cap: int) -> int:
    return int(lib().instant_calib_workspace_bytes(L, r_cap))


@dataclasses.dataclass
class CalibResult:
    k: int
    R: int
    scale: float
    energy: float
    eigenvalues: list


def calib_solve(C: torch.Tensor, n_samples: int, rows_out: torch.Tensor, *, eps: float = 0.95,
                p: int = 0, r_override: int = 0, scale_on: bool = True, max_iter: int = 0,
                tol: float = 0.0, ws: torch.Tensor | None = None, stream=None,
                raise_on_error: bool = True, warm_start: bool = False):
    """Projector rows from an accumulated statistic; synchronises the stream.

    With ``warm_start`` the rows already in ``rows_out`` (a previous projector
    of the same statistic) seed the eigensolver.

    Returns a :class:`CalibResult` (and the raw status when ``raise_on_error``
    is False)."""
    L = C.shape[0]
    r_cap = rows_out.shape[0]
    if C.shape != (L, L) or C.dtype != torch.float32 or rows_out.shape[1] != L:
        raise ValueError("calib_solve: inconsistent shapes")
    if ws is None:
        ws = torch.empty(calib_workspace_bytes(L, r_cap), dtype=torch.uint8, device=C.device)
    prm = CalibParams(eps, p, r_override, int(bool(scale_on)), max_iter, tol, int(bool(warm_start)))
    k = ctypes.c_int(0)
    R = ctypes.c_int(0)
    s = ctypes.c_float(0)
    E = ctypes.c_double(0)
    eig = (ctypes.c_double * r_cap)()
    st = lib().instant_calib_solve(_dev(C, "C"), int(n_samples), L, ctypes.byref(prm),
                                   _dev(rows_out, "rows_out"), r_cap, dtype_code(rows_out.dtype),
                                   ctypes.byref(k), ctypes.byref(R), ctypes.byref(s),
                                   ctypes.byref(E), eig, _dev(ws, "ws"),
                                   ws.numel() * ws.element_size(), _stream(stream))
    res = CalibResult(k.value, R.value, s.value, E.value, list(eig))
    if raise_on_error:
        check(st, "instant_calib_solve")
        return res
    return res, st


def calib_batch_workspace_bytes(L: int, count: int) -> int:
    return int(lib().instant_calib_batch_workspace_bytes(L, count))


def calib_solve_batch(problems, *, ws: torch.Tensor | None = None, stream=None,
                      raise_on_error: bool = True):
    """Several statistics of one token length in one call; synchronises the stream.

    ``problems`` is a sequence of dicts with the keys ``C`` (``[L, L]`` fp32),
    ``n_samples`` and ``rows_out`` (``[r_cap, L]``, one dtype for all), and
    optionally the keyword parameters of :func:`calib_solve` (``eps``, ``p``,
    ``r_override``, ``scale_on``, ``max_iter``, ``tol``, ``warm_start``).
    Returns a list of :class:`CalibResult` (and the list of per-problem
    statuses when ``raise_on_error`` is False)."""
    n = len(problems)
    if n < 1:
        raise ValueError("calib_solve_batch: no problems")
    L = problems[0]["C"].shape[0]
    dt = problems[0]["rows_out"].dtype
    arr = (CalibProblem * n)()
    eigs = []
    for i, q in enumerate(problems):
        C, rows = q["C"], q["rows_out"]
        if C.shape != (L, L) or C.dtype != torch.float32 or rows.shape[1] != L or rows.dtype != dt:
            raise ValueError("calib_solve_batch: inconsistent shapes or dtypes")
        r_cap = rows.shape[0]
        eig = (ctypes.c_double * r_cap)()
        eigs.append(eig)
        prm = CalibParams(q.get("eps", 0.95), q.get("p", 0), q.get("r_override", 0),
                          int(bool(q.get("scale_on", True))), q.get("max_iter", 0), q.get("tol", 0.0),
                          int(bool(q.get("warm_start", False))))
        arr[i] = CalibProblem(_dev(C, "C"), int(q["n_samples"]), prm, _dev(rows, "rows_out"), r_cap,
                              ctypes.cast(eig, ctypes.POINTER(ctypes.c_double)), 0, 0, 0.0, 0.0, 0)
    if ws is None:
        ws = torch.empty(calib_batch_workspace_bytes(L, n), dtype=torch.uint8,
                         device=problems[0]["C"].device)
    st = lib().instant_calib_solve_batch(arr, n, L, dtype_code(dt), _dev(ws, "ws"),
                                         ws.numel() * ws.element_size(), _stream(stream))
    res = [CalibResult(arr[i].k, arr[i].R, arr[i].scale, arr[i].energy, list(eigs[i]))
           for i in range(n)]
    if raise_on_error:
        check(st, "instant_calib_solve_batch")
        return res
    return res, [arr[i].status for i in range(n)]


class CalibBatch:
    """The same statistics solved together again and again (a layer's C_X into
    P and C_G into Q, every N_t steps): the argument block of
    ``instant_calib_solve_batch`` is built once; :meth:`solve` updates the
    sample counts and the warm-start flag and passes it.  The tensors given
    here must stay alive and in place."""

    def __init__(self, problems, ws: torch.Tensor):
        self.n = len(problems)
        if self.n < 1:
            raise ValueError("CalibBatch: no problems")
        self.L = problems[0]["C"].shape[0]
        self.dt = problems[0]["rows_out"].dtype
        self.arr = (CalibProblem * self.n)()
        self.eigs = []
        for i, q in enumerate(problems):
            C, rows = q["C"], q["rows_out"]
            if (C.shape != (self.L, self.L) or C.dtype != torch.float32 or rows.shape[1] != self.L
                    or rows.dtype != self.dt):
                raise ValueError("CalibBatch: inconsistent shapes or dtypes")
            eig = (ctypes.c_double * rows.shape[0])()
            self.eigs.append(eig)
            prm = CalibParams(q.get("eps", 0.95), q.get("p", 0), q.get("r_override", 0),
                              int(bool(q.get("scale_on", True))), q.get("max_iter", 0),
                              q.get("tol", 0.0), 0)
            self.arr[i] = CalibProblem(_dev(C, "C"), 1, prm, _dev(rows, "rows_out"), rows.shape[0],
                                       ctypes.cast(eig, ctypes.POINTER(ctypes.c_double)), 0, 0, 0.0,
                                       0.0, 0)
        need = calib_batch_workspace_bytes(self.L, self.n)
        if ws.numel() * ws.element_size() < need:
            raise ValueError("CalibBatch: workspace too small")
        self.ws_ptr = _dev(ws, "ws")
        self.ws_bytes = ws.numel() * ws.element_size()
        self.dcode = dtype_code(self.dt)

    def solve(self, n_samples, warm_start: bool = False, r_override=None, stream=None):
        """Solves every problem (``n_samples[i]`` samples in statistic i);
        ``r_override``: optional per-problem overrides.  Returns the list of
        :class:`CalibResult`; raises on the first failing problem."""
        for i in range(self.n):
            q = self.arr[i]
            q.n_samples = int(n_samples[i])
            q.prm.warm_start = int(bool(warm_start))
            if r_override is not None:
                q.prm.r_override = int(r_override[i])
        st = lib().instant_calib_solve_batch(self.arr, self.n, self.L, self.dcode, self.ws_ptr,
                                             self.ws_bytes, _stream(stream))
        check(st, "instant_calib_solve_batch")
        return [CalibResult(self.arr[i].k, self.arr[i].R, self.arr[i].scale, self.arr[i].energy,
                            list(self.eigs[i])) for i in range(self.n)]


def reconstruction_error(t: torch.Tensor, Q: torch.Tensor, S: torch.Tensor, ws: torch.Tensor,
                         stream=None) -> tuple[float, float]:
    """``(sum_b ||t_b - Q^T S_b||^2, sum_b ||t_b||^2)`` for ``S = Q t`` per sample
    (t ``[B, L, C]``, Q ``[R, L]``, S ``[B*R, C]``); synchronises the stream.
    ``ws`` is at least 16 bytes of device scratch."""
    B, L, C = t.shape
    R = Q.shape[0]
    if Q.shape != (R, L) or S.shape != (B * R, C):
        raise ValueError("reconstruction_error: inconsistent shapes")
    _same_dtype(t.dtype, ("Q", Q), ("S", S))
    e2 = ctypes.c_double(0)
    n2 = ctypes.c_double(0)
    check(lib().instant_reconstruction_error(_dev(t, "t"), _dev(Q, "Q"), _dev(S, "S"), B, L, C, R,
                                             dtype_code(t.dtype), ctypes.byref(e2),
                                             ctypes.byref(n2), _dev(ws, "ws"),
                                             ws.numel() * ws.element_size(), _stream(stream)),
          "instant_reconstruction_error")
    return e2.value, n2.value


def device_status(clear: bool = True, stream=None) -> int:
    """Sticky device-side status (0 when no bounded wait ran out)."""
    return int(lib().instant_device_status(int(clear), _stream(stream)))
