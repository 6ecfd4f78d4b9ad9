"""ctypes view of ``libfa_gb300.so`` (the C ABI of include/fa_gb300.h).

Argument marshalling only. The library is built in-tree by
``attention_fa2_attn_gb300.build``. If it is missing, loading fails loudly:
there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

_HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa_gb300.h")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_BOUNDS = 5

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_ULL = ctypes.c_ulonglong

# name -> (restype, argtypes); mirrors include/fa_gb300.h
SIGNATURES = {
    "fa_version": (_I, []),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_last_cuda_error_string": (ctypes.c_char_p, []),
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_f32": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "fa_bwd_workspace_bytes": (_SZ, [_I, _I, _I]),
    "fa_fwd_kv_outer": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P]),
    "fa_fwd_kv_outer_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "fa_num_splits_heuristic": (_I, [_I, _I, _I, _I]),
    "fa_num_splits_prefill": (_I, [_I, _I, _I, _I, _I, _I]),
    "fa_decode_num_splits": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "fa_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "fa_decode_splitkv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P]),
    "fa_decode_splitkv_static": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "fa_lse_merge": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "fa_decode_paged": (
        _I,
        [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P],
    ),
    "fa_get_last_device_error": (_I, [_P, ctypes.POINTER(_I)]),
    "fa_set_wait_timeout_ns": (None, [_ULL]),
    "fa_get_wait_timeouts": (None, [ctypes.POINTER(_ULL), ctypes.POINTER(_ULL)]),
    "fa_selftest_wait_timeout": (_I, [_ULL, _P]),
}

_lib = None


def header_symbols() -> list[str]:
    """Names of every function the public header declares."""
    text = open(_HEADER).read()
    return sorted(set(re.findall(r"^FA_API\s+[\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)))


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the CUDA library and bind its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if build_if_missing and _build.needs_build():
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing; build it with attention_fa2_attn_gb300.build.build()")
    l = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(l, name)
        f.restype = res
        f.argtypes = args
    _lib = l
    return l


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        l = lib()
        msg = l.fa_status_string(status).decode()
        if status == FA_ERR_CUDA:
            msg += ": " + l.fa_last_cuda_error_string().decode()
        super().__init__(f"{where}: {msg}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != FA_OK:
        raise FAError(status, where)
