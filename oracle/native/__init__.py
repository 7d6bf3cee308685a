"""The C++ FP64 oracle (oracle/moe_oracle.cpp) through ctypes (test
infrastructure only; see the oracle package notes).

Same module and function names as the numpy oracle (``formats``, ``quant``,
``layer``, ``lru``), so every pin runs against both; the numpy one stays as a
cross-check.  The arithmetic is all in the C++ library: this package only
marshals arrays and sequences its calls.  Build with ``python -m oracle.build``
(``__graft_entry__.build()`` does it); importing a module raises if the
library is missing.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .. import build as _build

_lib = None

_D = C.POINTER(C.c_double)
_F = C.POINTER(C.c_float)
_U8 = C.POINTER(C.c_uint8)
_I = C.POINTER(C.c_int)
_LL = C.POINTER(C.c_longlong)
_ULL = C.POINTER(C.c_ulonglong)

_SIGS = {
    "orc_set_threads": ([C.c_int], None),
    "orc_threads": ([], C.c_int),
    "orc_e2m1": ([C.c_int], C.c_double),
    "orc_e8m0": ([C.c_int], C.c_double),
    "orc_e4m3": ([C.c_int], C.c_double),
    "orc_dequant": ([_U8, _U8, C.c_int, C.c_int, C.c_int, C.c_float, _D], None),
    "orc_e2m1_encode_n": ([_D, C.c_longlong, _U8], None),
    "orc_e4m3_encode_n": ([_D, C.c_longlong, _U8], None),
    "orc_silu_n": ([_D, C.c_longlong, _D], None),
    "orc_quant_mxfp4": ([_F, C.c_int, C.c_int, _U8, _U8], None),
    "orc_quant_nvfp4": ([_F, C.c_int, C.c_int, C.c_float, _U8, _U8], None),
    "orc_quant_mxfp8": ([_F, C.c_int, C.c_int, _U8, _U8], None),
    "orc_round_bf16_n": ([_D, C.c_longlong, _D], None),
    "orc_act_roundtrip": ([_D, C.c_int, C.c_int, C.c_int, C.c_float, _D], None),
    "orc_router": ([_D, _F, _F, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, _I, _D, _D], None),
    "orc_permute": ([_I, C.c_int, C.c_int, C.c_int, _LL, _LL, _LL, _LL], None),
    "orc_expert_ffn": ([_D, C.c_int, C.c_int, C.c_int, _D, _D, _D, C.c_int, C.c_int, C.c_float, C.c_float, _D],
                       None),
    "orc_combine": ([_D, _D, _LL, C.c_int, C.c_int, C.c_int, _D, _D], None),
    "orc_lru_new": ([C.c_int, C.c_int], C.c_void_p),
    "orc_lru_free": ([C.c_void_p], None),
    "orc_lru_install": ([C.c_void_p, C.c_int, C.c_int], None),
    "orc_lru_step": ([C.c_void_p, _I, C.c_int, _I, _I, _I, _I], C.c_int),
    "orc_lru_state": ([C.c_void_p, _I, _ULL, _ULL, _I], None),
    "orc_lru_set": ([C.c_void_p, _I, _ULL, C.c_ulonglong], None),
    "orc_lru_resize": ([C.c_void_p, C.c_int], None),
}


def lib():
    global _lib
    if _lib is None:
        path = _build.lib_path()
        if not os.path.exists(path):
            raise RuntimeError("the C++ oracle is not built (expected %s); run `python -m oracle.build`" % path)
        L = C.CDLL(path)
        for name, (argt, rest) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = argt
            fn.restype = rest
        _lib = L
    return _lib


def arr(a, dtype):
    """Contiguous copy (or view) of ``a`` with ``dtype``."""
    return np.ascontiguousarray(a, dtype=dtype)


def ptr(a, ctype):
    return a.ctypes.data_as(C.POINTER(ctype))


def set_threads(n: int) -> None:
    """Threads of the oracle's parallel loops (0 = every core OpenMP sees)."""
    lib().orc_set_threads(int(n))


def threads() -> int:
    return int(lib().orc_threads())


from . import formats, quant, layer, lru  # noqa: E402,F401
