"""ctypes loader for libusp.so (the C ABI declared in include/usp.h).

Loading never falls back to anything: if the shared library is missing or
lacks a symbol, :func:`lib` raises.  ``build()`` in ``build.py`` produces it.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libusp.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "usp.h")

USP_OK = 0
USP_ERR_INVALID_ARG = 1
USP_ERR_DIVISIBILITY = 2
USP_ERR_UNSUPPORTED = 3
USP_ERR_WORKSPACE = 4
USP_ERR_CUDA = 5
USP_ERR_TIMEOUT = 6

USP_F32 = 0
USP_BF16 = 1
USP_MATERIALISED = 0
USP_FUSED = 1

_i64 = ctypes.c_int64
_int = ctypes.c_int
_vp = ctypes.c_void_p
_fp = ctypes.c_void_p  # float* passed as an address
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

SIGNATURES = {
    "usp_relayout_tok2head": (_int, [_vp, _vp, _i64, _i64, _i64, _i64, _int, _int, _int, _vp]),
    "usp_relayout_head2tok": (_int, [_vp, _vp, _i64, _i64, _i64, _i64, _int, _int, _int, _vp]),
    "usp_attn_chunk_fwd": (_int, [_vp, _vp, _vp, _vp, _fp, _i64, _i64, _i64, _i64, _i64, _f32, _int, _vp]),
    "usp_lse_merge": (_int, [_vp, _fp, _int, _vp, _fp, _i64, _i64, _i64, _i64, _int, _vp]),
    "usp_attention_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64, _int, _int, _int, _int, _int]),
    "usp_attention_fwd": (_int, [_vp, _vp, _vp, _vp, _fp, _i64, _i64, _i64, _i64, _int, _int, _f32, _int, _int,
                                 _vp, _sz, _vp]),
    "usp_attention_bwd": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, _int,
                                 _f32, _int, _vp, _sz, _vp]),
    "usp_attention_bwd_materialised": (_int, [_vp, _vp, _vp, _vp, _fp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                              _int, _int, _f32, _int, _vp, _sz, _vp]),
    "usp_attention_joint_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64, _i64, _int, _int, _int, _int, _int]),
    "usp_attention_fwd_joint": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _fp, _vp, _fp, _i64, _i64, _i64, _i64,
                                       _i64, _int, _int, _f32, _int, _int, _vp, _sz, _vp]),
    "usp_cross_attention_fwd": (_int, [_vp, _vp, _vp, _vp, _fp, _i64, _i64, _i64, _i64, _i64, _int, _int, _f32,
                                       _int, _vp]),
    "usp_quantize_e4m3": (_int, [_vp, _vp, _fp, _i64, _i64, _i64, _i64, _int, _int, _vp]),
    "usp_attention_fp8_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64, _int, _int]),
    "usp_attention_fwd_fp8": (_int, [_vp, _vp, _vp, _vp, _fp, _i64, _i64, _i64, _i64, _int, _int, _f32, _vp, _sz,
                                     _vp]),
    "usp_attention_fwd_noalloc": (_int, [_vp, _vp, _vp, _vp, _fp, _i64, _i64, _i64, _i64, _int, _int, _f32, _int,
                                         _vp]),
    "usp_device_status": (_int, [_vp]),
    "usp_status_string": (ctypes.c_char_p, [_int]),
    "usp_last_cuda_error": (_int, []),
    "usp_set_debug_spin_limit": (None, [ctypes.c_longlong]),
    "usp_set_spin_limit": (None, [ctypes.c_longlong]),
    "usp_profile_phases": (_int, [_int]),
    "usp_profile_read": (_int, [ctypes.POINTER(ctypes.c_float), _int]),
}

_LIB = None


class UspError(RuntimeError):
    def __init__(self, fn: str, status: int):
        name = _LIB.usp_status_string(status).decode() if _LIB is not None else str(status)
        extra = ""
        if status == USP_ERR_CUDA and _LIB is not None:
            extra = f" (cudaError {_LIB.usp_last_cuda_error()})"
        super().__init__(f"{fn} failed: {name}{extra}")
        self.status = status


def header_symbols() -> list[str]:
    """Function names declared in include/usp.h."""
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"\b(usp_[a-z0-9_]+)\s*\(", txt)))


def lib():
    """Load libusp.so and bind every entry point; raise if anything is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libusp.so not found at {LIB_PATH}; build it with "
            "`python -m diffusion_transformer_sequence_gb300.build` (there is no fallback path)")
    handle = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)  # AttributeError if the symbol is missing
        fn.restype = res
        fn.argtypes = args
    _LIB = handle
    return _LIB


def check(fn: str, status: int) -> None:
    if status != USP_OK:
        raise UspError(fn, status)
