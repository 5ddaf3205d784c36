"""ctypes loader of ``libinstant.so`` with the C prototypes of include/instant.h.

Argument marshalling only.  There is no fallback: if the shared object is
missing the import of any entry point raises.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libinstant.so")

INSTANT_F32 = 0
INSTANT_BF16 = 1

# size of the library's fixed g_hat_x array (INSTANT_GRAD_X_STATIC_SCRATCH_BYTES)
GRAD_X_STATIC_SCRATCH_BYTES = 8 << 20

STATUS_NAMES = {
    0: "INSTANT_OK",
    1: "INSTANT_ERR_ARG",
    2: "INSTANT_ERR_SHAPE",
    3: "INSTANT_ERR_DTYPE",
    4: "INSTANT_ERR_ALIGN",
    5: "INSTANT_ERR_WORKSPACE",
    6: "INSTANT_ERR_CUDA",
    7: "INSTANT_ERR_NOT_CONVERGED",
    8: "INSTANT_ERR_NONFINITE",
    9: "INSTANT_ERR_DEVICE",
}


class CalibParams(ctypes.Structure):
    _fields_ = [
        ("eps", ctypes.c_double),
        ("p", ctypes.c_int),
        ("r_override", ctypes.c_int),
        ("scale_on", ctypes.c_int),
        ("max_iter", ctypes.c_int),
        ("tol", ctypes.c_double),
        ("warm_start", ctypes.c_int),
    ]


class AccumulateItem(ctypes.Structure):
    _fields_ = [
        ("t", ctypes.c_void_p),
        ("C", ctypes.c_void_p),
        ("B", ctypes.c_int),
        ("Cdim", ctypes.c_int),
    ]


class CalibProblem(ctypes.Structure):
    _fields_ = [
        ("C", ctypes.c_void_p),
        ("n_samples", ctypes.c_longlong),
        ("prm", CalibParams),
        ("rows_out", ctypes.c_void_p),
        ("r_cap", ctypes.c_int),
        ("eig_out", ctypes.POINTER(ctypes.c_double)),
        ("k", ctypes.c_int),
        ("R", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("energy", ctypes.c_double),
        ("status", ctypes.c_int),
    ]


class InstantError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().instant_status_string(status).decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({msg})")


_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t

_PROTOS = {
    "instant_compress_act": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "instant_project_grad": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    "instant_grad_w": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    "instant_grad_x": (_i, [_vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _i, _vp]),
    "instant_grad_x_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "instant_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _i, _vp]),
    "instant_forward_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "instant_grad_w_x": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _i,
                              _i, _vp]),
    "instant_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _sz, _i, _i, _i, _i,
                              _i, _i, _i, _vp]),
    "instant_backward_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "instant_grad_x_core": (_i, [_vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _vp]),
    "instant_expand": (_i, [_vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _i, _vp]),
    "instant_grad_x_static": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    "instant_calib_accumulate": (_i, [_vp, _vp, _i, _i, _i, _i, _vp]),
    "instant_calib_accumulate_batch": (_i, [ctypes.POINTER(AccumulateItem), _i, _i, _i, _vp]),
    "instant_calib_solve": (_i, [_vp, ctypes.c_longlong, _i, ctypes.POINTER(CalibParams), _vp, _i,
                                 _i, ctypes.POINTER(_i), ctypes.POINTER(_i),
                                 ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double),
                                 ctypes.POINTER(ctypes.c_double), _vp, _sz, _vp]),
    "instant_calib_workspace_bytes": (_sz, [_i, _i]),
    "instant_calib_solve_batch": (_i, [ctypes.POINTER(CalibProblem), _i, _i, _i, _vp, _sz, _vp]),
    "instant_calib_batch_workspace_bytes": (_sz, [_i, _i]),
    "instant_reconstruction_error": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i,
                                          ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(ctypes.c_double), _vp, _sz, _vp]),
    "instant_device_status": (_i, [_i, _vp]),
    "instant_status_string": (ctypes.c_char_p, [_i]),
    "instant_version": (_i, []),
    "instant_launch_count": (ctypes.c_ulonglong, []),
}

_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises when it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(rank_compressed_backprop_gb300.build.build())")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _PROTOS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def check(status: int, where: str) -> None:
    if status != 0:
        raise InstantError(status, where)
