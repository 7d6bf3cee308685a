"""FP4 activation quantisers of the prefill regime, by the C++ oracle, with
the numpy oracle's names (fp32 decisions; see oracle/quant.py for the
reading).  Test infrastructure only."""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import arr, lib, ptr


def e2m1_encode(q: np.ndarray) -> np.ndarray:
    q = arr(q, np.float64)
    out = np.empty(q.shape, dtype=np.uint8)
    lib().orc_e2m1_encode_n(ptr(q, C.c_double), q.size, ptr(out, C.c_uint8))
    return out


def e4m3_encode_satfinite(v: np.ndarray) -> np.ndarray:
    v = arr(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_n(ptr(v, C.c_double), v.size, ptr(out, C.c_uint8))
    return out


def quant_mxfp4(v: np.ndarray):
    """(packed codes uint8 [rows, K/2], E8M0 bytes [rows, K/32]) of rows v."""
    v32 = arr(v, np.float32)
    rows, K = v32.shape
    codes = np.empty((rows, K // 2), dtype=np.uint8)
    scales = np.empty((rows, K // 32), dtype=np.uint8)
    lib().orc_quant_mxfp4(ptr(v32, C.c_float), rows, K, ptr(codes, C.c_uint8), ptr(scales, C.c_uint8))
    return codes, scales


def quant_nvfp4(v: np.ndarray, g: float):
    """(packed codes uint8 [rows, K/2], E4M3 bytes [rows, K/16]) of rows v."""
    v32 = arr(v, np.float32)
    rows, K = v32.shape
    codes = np.empty((rows, K // 2), dtype=np.uint8)
    scales = np.empty((rows, K // 16), dtype=np.uint8)
    lib().orc_quant_nvfp4(ptr(v32, C.c_float), rows, K, float(np.float32(g)), ptr(codes, C.c_uint8),
                          ptr(scales, C.c_uint8))
    return codes, scales


def quant_mxfp8(v: np.ndarray):
    """(E4M3 bytes uint8 [rows, K], E8M0 bytes [rows, K/32]) of rows v."""
    v32 = arr(v, np.float32)
    rows, K = v32.shape
    codes = np.empty((rows, K), dtype=np.uint8)
    scales = np.empty((rows, K // 32), dtype=np.uint8)
    lib().orc_quant_mxfp8(ptr(v32, C.c_float), rows, K, ptr(codes, C.c_uint8), ptr(scales, C.c_uint8))
    return codes, scales


def round_bf16(v: np.ndarray) -> np.ndarray:
    """v rounded to fp32, then to bf16 (each nearest even), as FP64."""
    v = arr(v, np.float64)
    out = np.empty(v.shape, dtype=np.float64)
    lib().orc_round_bf16_n(ptr(v, C.c_double), v.size, ptr(out, C.c_double))
    return out
