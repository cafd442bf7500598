"""Prox two-stage sparse SwiGLU FFN decode path for NVIDIA B300 (sm_103a).

Stage 1: input sparsity + INT4 proxies of W_gate and W_up -> salience -> one shared top-k
channel mask. Stage 2: exact bf16 gate/up/down projections over the masked channels only.
The kernels live in lib/libprox.so behind the C ABI of include/prox.h; this package is a
thin binding with the same function names.
"""
from .api import *  # noqa: F401,F403
from .api import __all__  # noqa: F401
from ._lib import LIB_PATH, lib  # noqa: F401
