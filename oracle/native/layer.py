"""One routed MoE layer forward pass in FP64 by the C++ oracle, with the numpy
oracle's names (router, permute, SwiGLU experts, combine, the Layer driver).
Test infrastructure only.

The arithmetic runs in oracle/moe_oracle.cpp (fixed-order loops, OpenMP over
tokens and rows); this module only marshals arrays and calls the steps in the
order the layer defines: router -> permute -> each routed expert on its rows
(+ the shared expert on every token) -> combine.  The definitions and the
readings are those of the numpy oracle (oracle/layer.py).
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, Optional, Sequence

import numpy as np

from . import arr, lib, ptr
from . import formats


def _fmt(fmt: str) -> int:
    return formats.FMT_ID[fmt]


def router(x, W_r, bias, k: int, norm_topk: bool = True):
    """(idx int32 [N, k] ascending, gates fp64 [N, k], logits fp64 [N, E])."""
    x = arr(x, np.float64)
    W = arr(W_r, np.float32)
    N, d = x.shape
    E = W.shape[0]
    b = None if bias is None else arr(bias, np.float32)
    idx = np.empty((N, k), dtype=np.int32)
    gates = np.empty((N, k), dtype=np.float64)
    L = np.empty((N, E), dtype=np.float64)
    lib().orc_router(ptr(x, C.c_double), ptr(W, C.c_float), None if b is None else ptr(b, C.c_float), N, d, E, k,
                     1 if norm_topk else 0, ptr(idx, C.c_int), ptr(gates, C.c_double), ptr(L, C.c_double))
    return idx, gates, L


def router_logits(x, W_r, bias) -> np.ndarray:
    return router(x, W_r, bias, 1)[2]


def near_tie(x, W_r, bias, k: int, thresh: float = 1e-4) -> np.ndarray:
    """True for tokens whose k-th and (k+1)-th largest FP64 logits differ by
    less than ``thresh``."""
    L = router_logits(x, W_r, bias)
    if k >= L.shape[1]:
        return np.zeros(L.shape[0], dtype=bool)
    s = -np.sort(-L, axis=1)
    return (s[:, k - 1] - s[:, k]) < thresh


def permute(idx: np.ndarray, E: int):
    """counts [E], offsets [E+1], row_of [N, k], tok_of [N*k] (int64)."""
    idx = arr(idx, np.int32)
    N, k = idx.shape
    counts = np.empty(E, dtype=np.int64)
    offsets = np.empty(E + 1, dtype=np.int64)
    row_of = np.empty((N, k), dtype=np.int64)
    tok_of = np.empty(N * k, dtype=np.int64)
    lib().orc_permute(ptr(idx, C.c_int), N, k, E, ptr(counts, C.c_longlong), ptr(offsets, C.c_longlong),
                      ptr(row_of, C.c_longlong), ptr(tok_of, C.c_longlong))
    return counts, offsets, row_of, tok_of


def silu(z: np.ndarray) -> np.ndarray:
    z = arr(z, np.float64)
    out = np.empty_like(z)
    lib().orc_silu_n(ptr(z, C.c_double), z.size, ptr(out, C.c_double))
    return out


def dequant_expert(w: Dict, fmt: str) -> Dict[str, np.ndarray]:
    """FP64 gate [f, d], up [f, d], down [d, f] of one expert."""
    return {n: formats.dequant(m.codes, m.scales, m.tscale, fmt) for n, m in w.items()}


def act_roundtrip(v: np.ndarray, fmt: str, g: float) -> np.ndarray:
    v = arr(v, np.float64)
    rows, K = v.shape
    out = np.empty_like(v)
    lib().orc_act_roundtrip(ptr(v, C.c_double), rows, K, _fmt(fmt), float(np.float32(g)), ptr(out, C.c_double))
    return out


def expert_ffn(X: np.ndarray, W: Dict[str, np.ndarray], regime: str = "decode", fmt: str = "mxfp4",
               g_x: float = 1.0, g_h: float = 1.0) -> np.ndarray:
    X = arr(X, np.float64)
    n, d = X.shape
    Wg, Wu, Wd = (arr(W[m], np.float64) for m in ("gate", "up", "down"))
    f = Wg.shape[0]
    out = np.empty((n, d), dtype=np.float64)
    lib().orc_expert_ffn(ptr(X, C.c_double), n, d, f, ptr(Wg, C.c_double), ptr(Wu, C.c_double),
                         ptr(Wd, C.c_double), 1 if regime == "prefill" else 0, _fmt(fmt),
                         float(np.float32(g_x)), float(np.float32(g_h)), ptr(out, C.c_double))
    return out


def combine(O: np.ndarray, gates: np.ndarray, row_of: np.ndarray, shared: Optional[np.ndarray] = None):
    O = arr(O, np.float64)
    gates = arr(gates, np.float64)
    row_of = arr(row_of, np.int64)
    N, k = gates.shape
    d = O.shape[1]
    sh = None if shared is None else arr(shared, np.float64)
    y = np.empty((N, d), dtype=np.float64)
    lib().orc_combine(ptr(O, C.c_double), ptr(gates, C.c_double), ptr(row_of, C.c_longlong), N, k, d,
                      None if sh is None else ptr(sh, C.c_double), ptr(y, C.c_double))
    return y


def _act_fmt(spec) -> str:
    """Activation format of the prefill regime: the weights' own format, or
    the spec's prefill_act (MXFP8 on MXFP4 weights: W4A8)."""
    return getattr(spec, "prefill_act", None) or spec.fmt


class Layer:
    """The layer's parameters as the oracle sees them: per-matrix FP4 arrays
    from the generator, dequantised on demand, one expert at a time."""

    def __init__(self, spec, experts_fn, router_w, router_b, shared_w=None, g_x: float = 1.0, g_h: float = 1.0):
        self.spec = spec
        self._experts_fn = experts_fn
        self.W_r = router_w
        self.b = router_b
        self.shared_w = shared_w
        self.g_x, self.g_h = g_x, g_h

    def expert(self, e: int) -> Dict[str, np.ndarray]:
        return dequant_expert(self._experts_fn(e), self.spec.fmt)

    def forward(self, x: np.ndarray, regime: str = "decode", tokens: Optional[Sequence[int]] = None):
        """FP64 y for the tokens ``tokens`` of x (all by default); (y, idx, gates)."""
        spec = self.spec
        x = arr(x, np.float64)
        if tokens is not None:
            x = x[np.asarray(tokens)]
        idx, gates, _ = router(x, self.W_r, self.b, spec.k, spec.norm_topk)
        counts, offsets, row_of, tok_of = permute(idx, spec.E)
        O = np.zeros((idx.size, spec.d_model), dtype=np.float64)
        for e in range(spec.E):
            if counts[e] == 0:
                continue
            rows = np.arange(offsets[e], offsets[e + 1])
            O[rows] = expert_ffn(x[tok_of[rows]], self.expert(e), regime, _act_fmt(spec), self.g_x, self.g_h)
        shared = None
        if spec.has_shared:
            shared = expert_ffn(x, dequant_expert(self.shared_w, spec.fmt), regime, _act_fmt(spec), self.g_x, self.g_h)
        return combine(O, gates, row_of, shared), idx, gates
