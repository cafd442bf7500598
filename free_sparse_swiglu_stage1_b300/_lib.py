"""ctypes view of libprox.so (include/prox.h). Loading fails loudly when the library is
missing: there is no fallback implementation."""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libprox.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "prox.h")


class ProxError(RuntimeError):
    """A libprox call returned an error code."""

    def __init__(self, code: int, where: str):
        self.code = code
        detail = ""
        if code == -3:   # PROX_ERR_CUDA: say which CUDA call failed and how
            try:
                detail = f" [{lib().prox_last_cuda_error().decode()}]"
            except Exception:
                pass
        super().__init__(f"{where}: {error_string(code)} ({code}){detail}")


class prox_cost_model(ctypes.Structure):
    _fields_ = [("in_cost", ctypes.c_double), ("fixed_cost", ctypes.c_double),
                ("ch_cost", ctypes.c_double), ("dense_cost", ctypes.c_double)]


class prox_packed(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("group", ctypes.c_int32), ("format", ctypes.c_int32),
                ("base", ctypes.c_void_p), ("bytes", ctypes.c_size_t),
                ("proxy", ctypes.c_void_p)]


_P = ctypes.POINTER(prox_packed)
_vp, _i, _d, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_float, ctypes.c_size_t

# name -> (restype, argtypes); must match include/prox.h
SIGNATURES = {
    "prox_packed_bytes": (_sz, [_i, _i, _i]),
    "prox_workspace_bytes": (_sz, [_i, _i, _i]),
    "prox_workspace_init": (_i, [_vp, _sz, _vp]),
    "prox_k_for": (_i, [_d, _i]),
    "prox_cost_model_bytes": (_i, [_i, _i, ctypes.POINTER(prox_cost_model)]),
    "prox_choose_sparsity": (_i, [ctypes.POINTER(prox_cost_model), _i, _i, _d, _d, _d, _vp, _vp,
                                  _vp]),
    "prox_pack_weights": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _sz, _vp, _P]),
    "prox_pack_weights_fp8": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _sz, _vp, _P]),
    "prox_packed_bytes_fp8": (_sz, [_i, _i, _i]),
    "prox_build_mask": (_i, [_P, _vp, _i, _d, _d, _vp, _vp, _sz, _vp]),
    "prox_sparse_ffn": (_i, [_P, _vp, _i, _vp, _i, _vp, _vp, _sz, _vp]),
    "prox_ffn_forward": (_i, [_P, _vp, _i, _d, _d, _vp, _vp, _vp, _sz, _vp]),
    "prox_ffn_forward_host": (_i, [_P, _vp, _i, _d, _d, _vp, _vp, _sz, _vp]),
    "prox_sparse_ffn_noalloc": (_i, [_P, _vp, _i, _vp, _i, _vp, _vp, _vp]),
    "prox_dense_ffn": (_i, [_P, _vp, _i, _vp, _vp, _sz, _vp]),
    "prox_rmsnorm": (_i, [_vp, _vp, _i, _i, _f, _vp]),
    "prox_get_status": (_i, [_vp, _vp]),
    "prox_error_string": (ctypes.c_char_p, [_i]),
    "prox_last_cuda_error": (ctypes.c_char_p, []),
    "prox_launch_count": (ctypes.c_uint64, []),
    "prox_debug_stage1": (_i, [_P, _vp, _i, _d, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "prox_debug_union": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "prox_debug_fused_forward": (_i, [_P, _vp, _d, _d, _vp, _vp, _vp, _sz, _vp]),
    "prox_debug_wait_timeout": (_i, [_vp, _sz, ctypes.c_longlong, _vp]),
    "prox_proxy_bytes": (_sz, [_i, _i, _i]),
    "prox_cost_model_fit": (_i, [_vp, _vp, _vp, _i, _d, _d, ctypes.POINTER(prox_cost_model)]),
    "prox_rows_bytes": (_sz, [_i, _i, _i, _i]),
    "prox_split_packed": (_i, [_P, _vp, _sz, _vp, _sz, _vp, _P]),
    "prox_window_create": (_i, [_i, _i, _i, _i, ctypes.POINTER(_vp), _vp, _sz,
                                ctypes.POINTER(_vp)]),
    "prox_window_acquire": (_i, [_vp, _i, _P, _vp]),
    "prox_window_release": (_i, [_vp, _i, _vp]),
    "prox_window_stats": (_i, [_vp, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
    "prox_window_destroy": (_i, [_vp]),
    "prox_debug_window_plan": (_i, [_i, _i, _vp, _i, _vp, _vp, _i, ctypes.POINTER(_i)]),
}

_lib: ctypes.CDLL | None = None


def header_symbols() -> list[str]:
    """Every function name include/prox.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b(prox_\w+)\s*\(", text, re.M)))


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"libprox.so not found at {LIB_PATH}; build it with "
                "`python -m free_sparse_swiglu_stage1_b300.build` (nvcc, sm_103a)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def error_string(code: int) -> str:
    try:
        return lib().prox_error_string(code).decode()
    except Exception:   # the library itself failed to load
        return f"error {code}"


def check(code: int, where: str) -> None:
    if code != 0:
        raise ProxError(code, where)
