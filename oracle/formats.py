"""FP4 weight formats, decoded in FP64 (oracle; test infrastructure only).

The FreeToken pages name the formats but do not define them: the GLM-5.2
checkpoint is NVFP4 and DeepSeek-V4-Flash is natively MXFP4 ("FreeToken：把
284B MoE 塞进游戏 PC", zhichai.net, §五), and the engine supports MXFP4, NVFP4,
FP8 and BF16 (juejin.cn overview, §五 模型生态与硬件支持).  The definitions
below are the public ones:

* E2M1 (OCP Microscaling Formats v1.0, FP4 element): sign bit 3, exponent
  bits 2..1 (bias 1), mantissa bit 0; exponent 0 is subnormal (0.5 * m).
* E8M0 (OCP MX v1.0 shared scale): 2^(x - 127); 255 is NaN (never drawn).
* E4M3 "fn" (OCP 8-bit FP, used as the NVFP4 block scale): bias 7,
  subnormals, no infinities, 0x7F / 0xFF NaN, max 448.
* MXFP4 = E2M1 elements, one E8M0 scale per 32 consecutive K elements.
* NVFP4 = E2M1 elements, one E4M3 scale per 16 K elements, one fp32 scale per
  tensor.
* MXFP8 (the "FP8" format, OCP MX v1.0) = E4M3 elements, one E8M0 scale per
  32 K elements.
* BF16 = the upper 16 bits of an IEEE fp32 value (sign, 8 exponent bits, 7
  mantissa bits), no scales.

Packing (pages silent; this build's layout): FP4 codes two per byte, the low
nibble holds the even K index; E4M3 codes one byte per element; bf16 elements
as little-endian byte pairs; scales are row-major [rows, K / block].
"""
from __future__ import annotations

import numpy as np


def e2m1_value(code: int) -> float:
    """Value of one 4-bit E2M1 code (OCP MX v1.0 FP4 element)."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if s else mag


def e8m0_value(x: int) -> float:
    """Value of an E8M0 scale byte: 2^(x-127); 255 is NaN."""
    if x == 255:
        return float("nan")
    return 2.0 ** (x - 127)


def e4m3_value(b: int) -> float:
    """Value of an E4M3 (fn) byte: bias 7, subnormals, 0x7F/0xFF NaN."""
    s = (b >> 7) & 1
    e = (b >> 3) & 15
    m = b & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E8M0_TABLE = np.array([e8m0_value(x) for x in range(256)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 [rows, K/2] -> uint8 codes [rows, K]; low nibble = even K."""
    out = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = codes & 0x0F
    out[:, 1::2] = codes >> 4
    return out


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """Values of bf16 bit patterns: the fp32 whose upper half they are."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def dequant(codes: np.ndarray, scales: np.ndarray, tscale: float, fmt: str) -> np.ndarray:
    """FP64 [rows, K] values of one weight matrix.

    MXFP4: w[r, i] = E2M1(c[r, i]) * E8M0(s[r, i // 32]).
    NVFP4: w[r, i] = E2M1(c[r, i]) * E4M3(s[r, i // 16]) * tscale.
    MXFP8: w[r, i] = E4M3(c[r, i]) * E8M0(s[r, i // 32]).
    BF16:  w[r, i] = bf16(bits of element i).
    """
    if fmt == "bf16":
        b = np.ascontiguousarray(codes, dtype=np.uint8)
        return bf16_value(b.view("<u2").reshape(b.shape[0], b.shape[1] // 2))
    if fmt == "mxfp8":
        vals = E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]
        return vals * np.repeat(E8M0_TABLE[scales], 32, axis=1)
    c = unpack_codes(codes)
    vals = E2M1_TABLE[c]
    if fmt == "mxfp4":
        block, stab, t = 32, E8M0_TABLE, 1.0
    elif fmt == "nvfp4":
        block, stab, t = 16, E4M3_TABLE, float(np.float32(tscale))
    else:
        raise ValueError(fmt)
    sc = np.repeat(stab[scales], block, axis=1)
    return vals * sc * t
