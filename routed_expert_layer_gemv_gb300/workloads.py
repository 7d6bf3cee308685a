"""Seeded synthetic workloads for one routed MoE layer.

This module only draws random inputs: packed FP4 code bytes, scale bytes,
normal hidden states and router weights.  It holds none of the layer's
arithmetic (no routing, no dequantisation, no FFN), so both the CUDA path and
the CPU oracle can take their inputs from it without sharing any of the
method's code.

Every tensor comes from its own substream: ``numpy.random.SeedSequence`` keyed
by ``(seed, tensor id, index...)`` feeding PCG64.  The same seed therefore
gives the same bytes on any machine, and one expert can be regenerated
without drawing the others (the CPU baseline draws only the experts a sample
touches).

The five layer shapes are those of the workloads the FreeToken pages measure
("FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §一 and §二: a 35B-A3B
model on consumer GPUs, a 284B-A13B DeepSeek-V4-Flash-class model and a 753B
GLM-5.2-class NVFP4 model).  The pages run trained checkpoints and replayed
agent traces; those are not available, so seeded draws of the same shapes
stand in for them.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Dict, Optional, Tuple

import numpy as np

MXFP4 = "mxfp4"
NVFP4 = "nvfp4"
MXFP8 = "mxfp8"
BF16 = "bf16"

# bits per weight code, and the K elements one block scale covers (0: none)
CODE_BITS = {MXFP4: 4, NVFP4: 4, MXFP8: 8, BF16: 16}
SCALE_BLOCK = {MXFP4: 32, NVFP4: 16, MXFP8: 32, BF16: 0}

# substream ids (one per tensor kind)
_SID_EXPERT = 1
_SID_SHARED = 2
_SID_ROUTER_W = 3
_SID_ROUTER_B = 4
_SID_X_IID = 5
_SID_X_AR1_INIT = 6
_SID_X_AR1_EPS = 7
_SID_REDRAW = 8


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """Shape of one routed MoE layer."""
    E: int                 # routed experts
    k: int                 # experts per token
    d_model: int
    d_ff: int
    n_slots: int           # expert-cache slots on the GPU
    fmt: str = MXFP4       # MXFP4 (E8M0 per 32), NVFP4 (E4M3 per 16 + fp32 per tensor),
                           # MXFP8 (E4M3 elements, E8M0 per 32) or BF16 (no scales)
    has_shared: bool = False
    has_bias: bool = False
    norm_topk: bool = True
    router_std: Optional[float] = None   # default 1/sqrt(d_model)
    bias_var: float = 0.5
    prefill_act: Optional[str] = None    # prefill activations: None = the weights' format;
                                         # MXFP8 on MXFP4 weights = W4A8

    @property
    def block(self) -> int:
        """K elements per block scale (0: the format has none)."""
        return SCALE_BLOCK[self.fmt]

    @property
    def act_fmt(self) -> str:
        """Format the prefill regime quantises x and h to."""
        return self.prefill_act or self.fmt


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layer: LayerSpec
    kind: str                      # "prefill" (one chunk) or "decode" (AR(1) steps)
    n_tokens: int = 0              # prefill chunk size
    batches: Tuple[int, ...] = ()  # decode tokens per step
    steps: int = 0                 # decode steps
    rho: float = 0.9
    seed: int = 0


# The five measured shapes.
TINY = Workload(
    "tiny_e8_top2_d256_f512_mxfp4",
    LayerSpec(E=8, k=2, d_model=256, d_ff=512, n_slots=8, fmt=MXFP4,
              router_std=1.0 / 16.0),
    kind="prefill", n_tokens=64)
DECODE_35B = Workload(
    "decode_35b_a3b_d2048_e128_top8_f768_mxfp4_s47",
    LayerSpec(E=128, k=8, d_model=2048, d_ff=768, n_slots=47, fmt=MXFP4),
    kind="decode", batches=(1, 4, 16), steps=512)
PREFILL_35B = Workload(
    "prefill_35b_a3b_n8192_d2048_e128_top8_f768_mxfp4",
    LayerSpec(E=128, k=8, d_model=2048, d_ff=768, n_slots=128, fmt=MXFP4),
    kind="prefill", n_tokens=8192)
DECODE_284B = Workload(
    "decode_284b_a13b_d4096_e256_top8_shared_f2048_mxfp4_s28",
    LayerSpec(E=256, k=8, d_model=4096, d_ff=2048, n_slots=28, fmt=MXFP4,
              has_shared=True),
    kind="decode", batches=(1, 8), steps=1024)
PREFILL_753B = Workload(
    "prefill_753b_n16384_d6144_e256_top8_shared_f2048_nvfp4_bias",
    LayerSpec(E=256, k=8, d_model=6144, d_ff=2048, n_slots=256, fmt=NVFP4,
              has_shared=True, has_bias=True),
    kind="prefill", n_tokens=16384)

WORKLOADS = [TINY, DECODE_35B, PREFILL_35B, DECODE_284B, PREFILL_753B]


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


# ---------------------------------------------------------------- bf16 bits

def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float64 draws to bf16 bit patterns (via fp32, each step
    round-to-nearest-even).  Input generation only."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- weights

@dataclasses.dataclass
class Matrix:
    """One weight matrix [rows, K], K contiguous.

    codes  uint8 [rows, K bits / 8]  MXFP4 / NVFP4: two E2M1 codes per byte,
                                     low nibble = even K; MXFP8: one E4M3 byte
                                     per element; BF16: the bf16 bits of each
                                     element, little-endian byte pairs
    scales uint8 [rows, K/B]         E8M0 (MXFP4, MXFP8: B=32) or E4M3 (NVFP4,
                                     B=16) bytes; [rows, 0] for BF16
    tscale float32                   per-tensor scale (NVFP4; 1.0 otherwise)
    """
    codes: np.ndarray
    scales: np.ndarray
    tscale: np.float32
    fmt: str = MXFP4

    @property
    def rows(self) -> int:
        return self.codes.shape[0]

    @property
    def K(self) -> int:
        return self.codes.shape[1] * 8 // CODE_BITS[self.fmt]


def _draw_matrix(g: np.random.Generator, rows: int, K: int, fmt: str) -> Matrix:
    if fmt == MXFP8:
        # E4M3 elements: random sign, exponent field 4..10 (values 2^-3 .. 15),
        # any mantissa; E8M0 exponent uniform over -10..-8 (biased 117..119):
        # a weight RMS near the FP4 formats'
        sgn = g.integers(0, 2, size=(rows, K), dtype=np.uint8)
        e = g.integers(4, 11, size=(rows, K), dtype=np.uint8)
        m = g.integers(0, 8, size=(rows, K), dtype=np.uint8)
        codes = ((sgn << 7) | (e << 3) | m).astype(np.uint8)
        scales = g.integers(127 - 10, 127 - 8 + 1, size=(rows, K // 32), dtype=np.uint8)
        return Matrix(codes, scales, np.float32(1.0), fmt)
    if fmt == BF16:
        # bf16 (RNE) of N(0, 0.05^2) draws
        bits = f64_to_bf16_bits(g.standard_normal((rows, K)) * 0.05)
        return Matrix(np.ascontiguousarray(bits).view(np.uint8).reshape(rows, 2 * K),
                      np.zeros((rows, 0), dtype=np.uint8), np.float32(1.0), fmt)
    # E2M1 codes uniform over all 16 values -> packed bytes uniform over 256
    codes = np.frombuffer(g.bytes(rows * (K // 2)), dtype=np.uint8).reshape(rows, K // 2).copy()
    if fmt == MXFP4:
        # E8M0 exponent uniform over the integers -8..-4 (biased 119..123)
        scales = g.integers(127 - 8, 127 - 4 + 1, size=(rows, K // 32), dtype=np.uint8)
        tscale = np.float32(1.0)
    else:
        # E4M3 block scale: positive normal codes, exponent field 4..8, any mantissa
        e = g.integers(4, 9, size=(rows, K // 16), dtype=np.uint8)
        m = g.integers(0, 8, size=(rows, K // 16), dtype=np.uint8)
        scales = ((e << 3) | m).astype(np.uint8)
        tscale = np.float32(2.0 ** -6)
    return Matrix(codes, scales, tscale, fmt)


def expert_weights(spec: LayerSpec, seed: int, e: int, shared: bool = False) -> Dict[str, Matrix]:
    """gate [f, d], up [f, d], down [d, f] of routed expert ``e`` (or the shared one)."""
    g = _rng(seed, _SID_SHARED if shared else _SID_EXPERT, e)
    d, f = spec.d_model, spec.d_ff
    return {
        "gate": _draw_matrix(g, f, d, spec.fmt),
        "up": _draw_matrix(g, f, d, spec.fmt),
        "down": _draw_matrix(g, d, f, spec.fmt),
    }


def router_weights(spec: LayerSpec, seed: int) -> Tuple[np.ndarray, Optional[np.ndarray]]:
    """W_r fp32 [E, d] ~ N(0, 1/d) (the variance reading), optional bias ~ N(0, 0.5)."""
    std = spec.router_std if spec.router_std is not None else 1.0 / np.sqrt(spec.d_model)
    W = (_rng(seed, _SID_ROUTER_W).standard_normal((spec.E, spec.d_model)) * std).astype(np.float32)
    b = None
    if spec.has_bias:
        b = (_rng(seed, _SID_ROUTER_B).standard_normal(spec.E) * np.sqrt(spec.bias_var)).astype(np.float32)
    return W, b


# ---------------------------------------------------------------- tokens

RejectFn = Callable[[np.ndarray], np.ndarray]


def iid_tokens(seed: int, n: int, d: int, reject: Optional[RejectFn] = None,
               max_redraws: int = 64) -> Tuple[np.ndarray, int]:
    """bf16 bits [n, d] of i.i.d. N(0,1) hidden states.

    ``reject(x_f64 [m, d]) -> bool [m]`` marks rows to redraw (the parity tests
    pass a near-tie detector); a redrawn row ``t`` takes attempt ``a`` from
    substream (seed, redraw, t, a).  Returns (bits, number of redraws).
    """
    x = f64_to_bf16_bits(_rng(seed, _SID_X_IID, n, d).standard_normal((n, d)))
    redraws = 0
    if reject is not None:
        bad = np.nonzero(reject(bf16_bits_to_f64(x)))[0]
        for t in bad:
            for a in range(max_redraws):
                row = f64_to_bf16_bits(_rng(seed, _SID_REDRAW, int(t), a).standard_normal(d))
                redraws += 1
                if not reject(bf16_bits_to_f64(row[None, :]))[0]:
                    x[t] = row
                    break
            else:
                raise RuntimeError("could not redraw token %d away from a near tie" % t)
    return x, redraws


def ar1_tokens(seed: int, batch: int, steps: int, d: int, rho: float = 0.9,
               reject: Optional[RejectFn] = None, max_redraws: int = 64) -> Tuple[np.ndarray, int]:
    """bf16 bits [steps, batch, d]: per batch row an independent AR(1) stream
    h_0 ~ N(0, I), h_t = rho h_{t-1} + sqrt(1 - rho^2) eps_t (unit variance);
    the token is bf16(h_t).  A rejected token redraws its innovation eps_t."""
    c = np.sqrt(1.0 - rho * rho)
    out = np.empty((steps, batch, d), dtype=np.uint16)
    redraws = 0
    for b in range(batch):
        h = _rng(seed, _SID_X_AR1_INIT, b, d).standard_normal(d)
        eps = _rng(seed, _SID_X_AR1_EPS, b, d).standard_normal((steps, d))
        for t in range(steps):
            ht = h if t == 0 else rho * h + c * eps[t]
            row = f64_to_bf16_bits(ht)
            if reject is not None and reject(bf16_bits_to_f64(row[None, :]))[0]:
                for a in range(max_redraws):
                    e2 = _rng(seed, _SID_REDRAW, 1_000_000 + b, t, a).standard_normal(d)
                    ht = (_rng(seed, _SID_REDRAW, 2_000_000 + b, t, a).standard_normal(d)
                          if t == 0 else rho * h + c * e2)
                    row = f64_to_bf16_bits(ht)
                    redraws += 1
                    if not reject(bf16_bits_to_f64(row[None, :]))[0]:
                        break
                else:
                    raise RuntimeError("could not redraw token (%d, %d) away from a near tie" % (t, b))
            out[t, b] = row
            h = ht
    return out, redraws
