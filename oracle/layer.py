"""One routed MoE layer forward pass in FP64 (oracle; test infrastructure only).

Pages.  The FreeToken pages describe decode as: the router picks a few experts
per token, most of them hit the GPU's LRU expert cache, the misses are filled
("FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §二 "Decode: q⋆ = m·B_P/B_H"
paragraph); expert routing varies per layer and per token (ananclaw.com
explainer, §核心方法 1); architectures differ in routing, expert count and the
presence of a shared expert (explainer, §核心方法 4).  They give no formula for
the layer, so each step below is the standard definition, with the reading
stated where a choice exists:

router   logits[t, e] = sum_i x[t, i] W_r[e, i] (+ b[e]); the k largest logits
         are selected (ties: lower expert index first, softmax is monotone so
         selecting on logits equals selecting on probabilities); gates are the
         softmax restricted to the selected logits (norm_topk, the plain
         reading for the named model families) or the full softmax
         probabilities (norm_topk = False).  The bias, when present, enters
         both the selection and the softmax.  Output order: ascending expert.
permute  counts[e], offsets = exclusive prefix sum over ascending e, and the
         rows of one expert in ascending token order (unique).
expert   out_e(x) = W_d (SiLU(W_g x) * (W_u x)), SiLU(z) = z / (1 + e^-z).
         Decode regime: x used as bf16-exact values.  Prefill regime: x and h
         pass through the block quantiser of the activation format first
         (``quant``): the weights' own format, or MXFP8 on MXFP4 weights
         (W4A8, the spec's ``prefill_act``).
combine  y[t] = sum_j g[t, j] out_{e_j}(x_t) + shared(x_t)  (shared expert
         always on, weight 1).
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

from . import formats, quant


# ------------------------------------------------------------------ router

def router_logits(x: np.ndarray, W_r: np.ndarray, bias: Optional[np.ndarray]) -> np.ndarray:
    """FP64 logits [N, E] from bf16-exact x [N, d] and fp32 W_r [E, d]."""
    L = np.asarray(x, np.float64) @ np.asarray(W_r, np.float64).T
    if bias is not None:
        L = L + np.asarray(bias, np.float64)[None, :]
    return L


def topk_select(L: np.ndarray, k: int) -> np.ndarray:
    """Indices [N, k] of the k largest logits per row (ties to the lower
    expert index), returned in ascending expert order."""
    N, E = L.shape
    # stable sort on -logit keeps equal logits in ascending index order
    order = np.argsort(-L, axis=1, kind="stable")[:, :k]
    return np.sort(order, axis=1)


def router(x, W_r, bias, k: int, norm_topk: bool = True):
    """Returns (idx int32 [N, k] ascending, gates fp64 [N, k], logits [N, E])."""
    L = router_logits(x, W_r, bias)
    idx = topk_select(L, k)
    m = L.max(axis=1, keepdims=True)
    p = np.exp(L - m)
    if norm_topk:
        sel = np.take_along_axis(p, idx, axis=1)
        gates = sel / sel.sum(axis=1, keepdims=True)
    else:
        p = p / p.sum(axis=1, keepdims=True)
        gates = np.take_along_axis(p, idx, axis=1)
    return idx.astype(np.int32), gates, L


def near_tie(x, W_r, bias, k: int, thresh: float = 1e-4) -> np.ndarray:
    """True for tokens whose k-th and (k+1)-th largest FP64 logits differ by
    less than ``thresh`` (such tokens are redrawn by the generator)."""
    L = router_logits(x, W_r, bias)
    if k >= L.shape[1]:
        return np.zeros(L.shape[0], dtype=bool)
    s = -np.sort(-L, axis=1)
    return (s[:, k - 1] - s[:, k]) < thresh


# ------------------------------------------------------------------ permute

def permute(idx: np.ndarray, E: int):
    """counts [E], offsets [E+1], row_of [N, k], tok_of [N*k]."""
    N, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for e in idx.reshape(-1):
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    fill = offsets[:-1].copy()
    row_of = np.empty((N, k), dtype=np.int64)
    tok_of = np.empty(N * k, dtype=np.int64)
    for t in range(N):              # ascending token order within each expert
        for j in range(k):
            e = idx[t, j]
            row_of[t, j] = fill[e]
            tok_of[fill[e]] = t
            fill[e] += 1
    return counts, offsets, row_of, tok_of


# ------------------------------------------------------------------ experts

def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def dequant_expert(w: Dict, fmt: str) -> Dict[str, np.ndarray]:
    """FP64 gate [f, d], up [f, d], down [d, f] of one expert."""
    return {n: formats.dequant(m.codes, m.scales, m.tscale, fmt) for n, m in w.items()}


def act_roundtrip(v: np.ndarray, fmt: str, g: float) -> np.ndarray:
    """The values the prefill activation quantiser hands to the MMA (FP64):
    the weight's block format (FP4 weights), MXFP8 (MXFP8 weights), bf16
    (BF16 weights)."""
    if fmt == "bf16":
        return quant.round_bf16(v)
    if fmt == "mxfp8":
        c, s = quant.quant_mxfp8(v)
        return formats.dequant(c, s, 1.0, "mxfp8")
    if fmt == "mxfp4":
        c, s = quant.quant_mxfp4(v)
        return formats.dequant(c, s, 1.0, "mxfp4")
    c, s = quant.quant_nvfp4(v, g)
    return formats.dequant(c, s, 1.0, "nvfp4") * float(np.float32(g))


def expert_ffn(X: np.ndarray, W: Dict[str, np.ndarray], regime: str = "decode",
               fmt: str = "mxfp4", g_x: float = 1.0, g_h: float = 1.0) -> np.ndarray:
    """SwiGLU expert on rows X [n, d] with dequantised weights W (FP64); in
    the prefill regime x and h are quantised to the activation format `fmt`."""
    X = np.asarray(X, np.float64)
    if regime == "prefill":
        X = act_roundtrip(X, fmt, g_x)
    a = X @ W["gate"].T
    u = X @ W["up"].T
    h = silu(a) * u
    if regime == "prefill":
        h = act_roundtrip(h, fmt, g_h)
    return h @ W["down"].T


# ------------------------------------------------------------------ combine

def combine(O: np.ndarray, gates: np.ndarray, row_of: np.ndarray,
            shared: Optional[np.ndarray] = None) -> np.ndarray:
    """y[t] = sum_j gates[t, j] O[row_of[t, j]] (+ shared[t])."""
    N, k = gates.shape
    y = np.zeros((N, O.shape[1]), dtype=np.float64)
    for j in range(k):
        y += gates[:, j:j + 1] * O[row_of[:, j]]
    if shared is not None:
        y = y + shared
    return y


# ------------------------------------------------------------------ layer

def _act_fmt(spec) -> str:
    """Activation format of the prefill regime: the weights' own format, or
    the spec's prefill_act (MXFP8 on MXFP4 weights: W4A8)."""
    return getattr(spec, "prefill_act", None) or spec.fmt


class Layer:
    """The layer's parameters as the oracle sees them: per-matrix FP4 arrays
    from the generator, dequantised on demand, one expert at a time."""

    def __init__(self, spec, experts_fn, router_w, router_b, shared_w=None,
                 g_x: float = 1.0, g_h: float = 1.0):
        self.spec = spec
        self._experts_fn = experts_fn     # e -> {"gate","up","down"} Matrix
        self.W_r = router_w
        self.b = router_b
        self.shared_w = shared_w
        self.g_x, self.g_h = g_x, g_h

    def expert(self, e: int) -> Dict[str, np.ndarray]:
        return dequant_expert(self._experts_fn(e), self.spec.fmt)

    def forward(self, x: np.ndarray, regime: str = "decode",
                tokens: Optional[Sequence[int]] = None):
        """FP64 y for the tokens ``tokens`` of x (all by default).

        Tokens are independent, so a subset gives the same values as the full
        batch (up to FP64 rounding order).  Returns (y [n, d], idx, gates)."""
        spec = self.spec
        x = np.asarray(x, np.float64)
        if tokens is not None:
            x = x[np.asarray(tokens)]
        idx, gates, _ = router(x, self.W_r, self.b, spec.k, spec.norm_topk)
        counts, offsets, row_of, tok_of = permute(idx, spec.E)
        O = np.zeros((idx.size, spec.d_model), dtype=np.float64)
        for e in range(spec.E):
            if counts[e] == 0:
                continue
            rows = np.arange(offsets[e], offsets[e + 1])
            O[rows] = expert_ffn(x[tok_of[rows]], self.expert(e), regime,
                                 _act_fmt(spec), self.g_x, self.g_h)
        shared = None
        if spec.has_shared:
            Ws = dequant_expert(self.shared_w, spec.fmt)
            shared = expert_ffn(x, Ws, regime, _act_fmt(spec), self.g_x, self.g_h)
        y = combine(O, gates, row_of, shared)
        return y, idx, gates
