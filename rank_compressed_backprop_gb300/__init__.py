"""GB300-native INSTANT low-rank backpropagation for linear layers.

The compute lives in ``libinstant.so`` (C ABI in include/instant.h, CUDA
kernels for sm_103a); this package is its Python binding.
"""

from . import api  # noqa: F401
from ._lib import InstantError, LIB_PATH, lib  # noqa: F401
from .layer import InstantLinear, LayerCalibration  # noqa: F401

__version__ = "0.1.0"
