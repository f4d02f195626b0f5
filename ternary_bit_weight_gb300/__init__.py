"""ternary_bit_weight_gb300: the ternary-weight linear layer on one GB300.

The product is libtern (C ABI, include/tern.h) with hand-written sm_103a
CUDA kernels; this package builds it in-tree and binds it with ctypes.
"""
from .binding import *  # noqa: F401,F403
from .binding import EXPORTED, TernError, library, library_path, status_string  # noqa: F401
