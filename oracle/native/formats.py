"""FP4 weight formats decoded in FP64 by the C++ oracle (OCP Microscaling
v1.0 E2M1 / E8M0, OCP 8-bit E4M3; MXFP4 and NVFP4 block layouts), with the
numpy oracle's names.  Test infrastructure only."""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import arr, lib, ptr


def e2m1_value(code: int) -> float:
    return float(lib().orc_e2m1(int(code)))


def e8m0_value(x: int) -> float:
    return float(lib().orc_e8m0(int(x)))


def e4m3_value(b: int) -> float:
    return float(lib().orc_e4m3(int(b)))


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E8M0_TABLE = np.array([e8m0_value(x) for x in range(256)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 [rows, K/2] -> uint8 codes [rows, K]; low nibble = even K."""
    out = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = codes & 0x0F
    out[:, 1::2] = codes >> 4
    return out


FMT_ID = {"mxfp4": 0, "nvfp4": 1, "mxfp8": 2, "bf16": 3}
_ELEMS_PER_BYTE = {"mxfp4": 2.0, "nvfp4": 2.0, "mxfp8": 1.0, "bf16": 0.5}


def dequant(codes: np.ndarray, scales: np.ndarray, tscale: float, fmt: str) -> np.ndarray:
    """FP64 [rows, K] of one weight matrix (C++ orc_dequant)."""
    c = arr(codes, np.uint8)
    s = arr(scales, np.uint8)
    rows, K = c.shape[0], int(c.shape[1] * _ELEMS_PER_BYTE[fmt])
    if s.size == 0:
        s = np.zeros(1, dtype=np.uint8)
    out = np.empty((rows, K), dtype=np.float64)
    lib().orc_dequant(ptr(c, C.c_uint8), ptr(s, C.c_uint8), rows, K, FMT_ID[fmt],
                      float(np.float32(tscale)), ptr(out, C.c_double))
    return out
