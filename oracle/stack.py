"""A stack of routed MoE layers sharing one GPU expert cache (oracle; test
infrastructure only).

Pages.  FreeToken keeps one LRU expert cache for the experts of every layer
("FreeToken：把 284B MoE 塞进游戏 PC", zhichai.net, §二, "LRU 为什么赢" paragraph;
juejin.cn overview, §二 全局 LRU 专家缓存), and in prefill it streams the experts
of a layer whole, the next layer's while the current one computes (zhichai.net
§二 "Prefill：把计算藏进传输"; juejin.cn §二 全层双缓冲预填充).  Readings taken:

* The stack is the layers' MoE sublayers in order: layer l's output, rounded
  to bf16 (the activation type between layers), is layer l + 1's input.  The
  rest of each transformer block (attention, norms, residuals) is out of scope.
* One table over all layers' experts: expert e of layer l is key l E + e, and
  each layer's step is the single-layer step (oracle.lru) on its keys -- hits
  first, misses ascending, the least recently used key of any layer evicted.
* Whole-layer prefetch (prefill): before layer l's own step, all E experts of
  layer l are accessed as one step by the same rule, so that step hits every
  routed expert.  Overlapped and serial prefetch give the same sequence of
  table steps: prefetch(0), step(0), prefetch(1), step(1), ...

The functions take the layers and the slot-table class as arguments, so the
same composition runs over either oracle implementation (numpy or C++).
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np


def bf16_round(v) -> np.ndarray:
    """Round FP64 values to the nearest bf16 value, ties to even (IEEE
    round-to-nearest-even onto the bf16 grid: 8 significant bits, exponent
    range of fp32, subnormal spacing 2^-133); overflow gives +-inf."""
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()
    fin = np.isfinite(v) & (v != 0.0)
    x = v[fin]
    _, e = np.frexp(x)                       # x = m 2^e, 0.5 <= |m| < 1
    q = np.maximum(e, -125) - 8              # spacing of bf16 values near x
    r = np.ldexp(np.rint(np.ldexp(x, -q)), q)
    big = np.abs(r) >= 2.0 ** 128
    r[big] = np.copysign(np.inf, x[big])
    out[fin] = r
    return out


def key(l: int, e: int, E: int) -> int:
    return l * E + e


def stack_forward(layers: Sequence, x, regime: str = "decode"):
    """Run the layers in order.  x: FP64 values (bf16-exact) [N, d].
    Returns (final hidden state as bf16 values, per-layer FP64 outputs,
    per-layer inputs, per-layer top-k ids)."""
    h = np.asarray(x, dtype=np.float64)
    ys, ins, ids = [], [], []
    for L in layers:
        ins.append(h)
        y, idx, _ = L.forward(h, regime)
        ys.append(y)
        ids.append(idx)
        h = bf16_round(y)
    return h, ys, ins, ids


class StackCache:
    """The stack's one slot table (n_slots slots over n_layers * E keys)."""

    def __init__(self, n_layers: int, E: int, S: int, table_cls):
        self.L, self.E, self.S = n_layers, E, S
        self.T = table_cls(n_layers * E, S)

    def step(self, l: int, routed: Sequence[int]) -> List[Tuple[int, int, bool, int]]:
        """Layer l's step on the experts `routed` (the layer's own ids);
        returns the access list with keys."""
        return self.T.step([key(l, int(e), self.E) for e in routed])

    def prefetch(self, l: int) -> List[Tuple[int, int, bool, int]]:
        """Every expert of layer l accessed as one step."""
        return self.T.step([key(l, e, self.E) for e in range(self.E)])

    @property
    def expert_of(self) -> List[int]:
        return list(self.T.expert_of)

    @property
    def stamp(self) -> List[int]:
        return list(self.T.stamp)

    @property
    def clock(self) -> int:
        return int(self.T.clock)
