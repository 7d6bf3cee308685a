"""Activation quantisers of the FP4 x FP4 prefill regime (oracle; test
infrastructure only).

The pages say the engine runs MXFP4 / NVFP4 checkpoints (zhichai.net §五;
juejin.cn §五) but not how activations meet FP4 weights.  Reading taken: the
prefill regime multiplies FP4 activations by FP4 weights (block-scaled FP4 MMA
needs both operands in FP4), so x before gate/up and h before down are
quantised to the weight's block format:

* MXFP4 (OCP MX v1.0 conversion): per 32 consecutive K elements, the shared
  exponent X = floor(log2(amax)) - 2 (2 = the largest E2M1 exponent), clamped
  to [-127, 127]; an all-zero block takes X = -127.  Elements are v / 2^X
  rounded to E2M1 (nearest, ties to the even code, saturating at 6).
* NVFP4: per 16 K elements the block scale is E4M3(amax / 6 / g), rounded to
  nearest-even and saturated at 448, where g is the layer's static fp32
  activation scale (a calibrated per-tensor scale, here a power of two);
  elements are v / (scale * g) rounded to E2M1.  A block whose scale is 0
  gets all-zero codes.

For the FP8 and BF16 weight formats (juejin.cn §五 lists FP8 and BF16 next to
the FP4 ones) the prefill regime's activations take the weight's element
type: MXFP8 weights meet MXFP8 activations (W8A8; OCP MX v1.0 conversion: per
32-block X = floor(log2(amax)) - 8 (8 = the largest E4M3 exponent), elements
v / 2^X rounded to E4M3, nearest even, saturating at 448), BF16 weights meet
bf16 activations (W16A16; v rounded to bf16, nearest even).

Where a floating-point value decides a code, the quotient is formed in fp32
(as the CUDA kernels form it), with IEEE round-to-nearest division, so both
sides take the same decision from the same input.  Rounding keeps the sign: a
negative value that rounds to zero encodes as -0 (code 8).
"""
from __future__ import annotations

import numpy as np

from .formats import E2M1_TABLE, E4M3_TABLE

_MAGS = E2M1_TABLE[:8]  # 0, .5, 1, 1.5, 2, 3, 4, 6 (codes 0..7)


def e2m1_encode(q: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code of each value (ties to the even code, saturating at
    +-6, sign kept).  Brute force over the 8 magnitudes."""
    q = np.asarray(q, dtype=np.float64)
    a = np.abs(q)
    dist = np.abs(a[..., None] - _MAGS)           # [..., 8]
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best
    # among equally near codes prefer the even one (there are at most two)
    even = cand & (np.arange(8) % 2 == 0)
    pick = np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(cand, axis=-1))
    pick = np.where(a >= 6.0, 7, pick)
    sign = np.signbit(q).astype(np.uint8)
    return (pick.astype(np.uint8) | (sign << 3)).astype(np.uint8)


_E4M3_POS = E4M3_TABLE[:0x7F]  # finite non-negative values, bytes 0..126


def e4m3_encode_satfinite(v: np.ndarray) -> np.ndarray:
    """Nearest non-negative finite E4M3 byte (ties to even mantissa, values
    above 448 saturate to 448).  Inputs are >= 0.  Brute force."""
    v = np.asarray(v, dtype=np.float64)
    dist = np.abs(v[..., None] - _E4M3_POS)
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best
    even = cand & (np.arange(0x7F) % 2 == 0)
    pick = np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(cand, axis=-1))
    pick = np.where(v >= 448.0, 0x7E, pick)
    return pick.astype(np.uint8)


def e4m3_encode_signed(q: np.ndarray) -> np.ndarray:
    """Nearest E4M3 byte of each value (ties to the even byte, magnitudes of
    448 and above saturate to 448, sign kept: -0 is 0x80)."""
    q = np.asarray(q, dtype=np.float64)
    mag = e4m3_encode_satfinite(np.abs(q))
    return (mag | (np.signbit(q).astype(np.uint8) << 7)).astype(np.uint8)


def quant_mxfp8(v: np.ndarray):
    """Quantise rows v [rows, K] (values exact in fp32) to MXFP8.

    Returns (E4M3 bytes uint8 [rows, K], E8M0 bytes [rows, K/32])."""
    v32 = np.asarray(v, dtype=np.float32)
    rows, K = v32.shape
    blk = v32.reshape(rows, K // 32, 32)
    amax = np.abs(blk).max(axis=-1).astype(np.float64)
    _, ex = np.frexp(amax)                          # amax = m * 2^ex, m in [0.5, 1)
    X = np.where(amax > 0, (ex - 1) - 8, -127)      # floor(log2 amax) - 8
    X = np.clip(X, -127, 127)
    q = (blk.astype(np.float64) * np.exp2(-X)[..., None]).astype(np.float32)   # exact (power of two)
    codes = e4m3_encode_signed(q.astype(np.float64)).reshape(rows, K)
    return codes, (X + 127).astype(np.uint8)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """v (FP64) rounded to fp32, then to bf16 (each nearest even): the bf16
    activations the W16A16 MMA takes (FP64 values)."""
    u = np.ascontiguousarray(np.asarray(v, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32)
    return (r << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def _pack(codes: np.ndarray) -> np.ndarray:
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def quant_mxfp4(v: np.ndarray):
    """Quantise rows v [rows, K] (values exact in fp32) to MXFP4.

    Returns (packed codes uint8 [rows, K/2], E8M0 bytes [rows, K/32])."""
    v32 = np.asarray(v, dtype=np.float32)
    rows, K = v32.shape
    blk = v32.reshape(rows, K // 32, 32)
    amax = np.abs(blk).max(axis=-1).astype(np.float64)
    _, ex = np.frexp(amax)                          # amax = m * 2^ex, m in [0.5, 1)
    X = np.where(amax > 0, (ex - 1) - 2, -127)      # floor(log2 amax) - 2
    X = np.clip(X, -127, 127)
    # v / 2^X in fp32: a power-of-two scaling, formed exactly
    q = (blk.astype(np.float64) * np.ldexp(1.0, -X)[..., None]).astype(np.float32)
    codes = e2m1_encode(q.astype(np.float64)).reshape(rows, K)
    return _pack(codes), (X + 127).astype(np.uint8)


def quant_nvfp4(v: np.ndarray, g: float):
    """Quantise rows v [rows, K] to NVFP4 with static activation scale g.

    Returns (packed codes uint8 [rows, K/2], E4M3 bytes [rows, K/16])."""
    v32 = np.asarray(v, dtype=np.float32)
    g32 = np.float32(g)
    rows, K = v32.shape
    blk = v32.reshape(rows, K // 16, 16)
    amax = np.abs(blk).max(axis=-1)                              # fp32
    s_raw = (amax / np.float32(6.0)) / g32                       # fp32, IEEE division
    sbyte = e4m3_encode_satfinite(s_raw.astype(np.float64))
    sval = E4M3_TABLE[sbyte].astype(np.float32)
    denom = (sval * g32).astype(np.float32)                      # exact: g is a power of two
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (blk / denom[..., None]).astype(np.float32)          # fp32, IEEE division
    q = np.where(denom[..., None] > 0, q, np.float32(0.0))
    codes = e2m1_encode(q.astype(np.float64)).reshape(rows, K)
    return _pack(codes), sbyte
