"""Pins of the stack oracle (oracle/stack.py) -- bf16 rounding between layers,
the one table keyed by (layer, expert), the whole-layer prefetch, the order
of the layers -- against torch's bf16 conversion, a naive list over
(layer, expert) pairs and a dense two-layer computation written out (no GPU)."""
import numpy as np
import pytest
import torch

from conftest import ORACLES, oracle_ns

from oracle import stack as ostack
from routed_expert_layer_gemv_gb300 import workloads as wl


@pytest.fixture(params=ORACLES)
def ns(request):
    return oracle_ns(request.param)


def test_bf16_round_matches_torch_conversion():
    # fp32 values are exact in FP64, and torch rounds fp32 -> bf16 to nearest even
    rng = np.random.default_rng(3)
    mags = np.ldexp(1.0, rng.integers(-140, 120, size=4000))
    v = (rng.standard_normal(4000) * mags).astype(np.float32)
    # ties between two bf16 values, both parities, and the subnormal range
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -130 + 2.0 ** -134,
                     3.0 * 2.0 ** -134, 2.0 ** -126 * (1 + 2.0 ** -8), 3.3895313892515355e38], np.float32)
    v = np.concatenate([v, ties, np.array([0.0, -0.0, np.inf, -np.inf], np.float32)])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = ostack.bf16_round(v.astype(np.float64))
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


class NaivePairLRU:
    """Recency as a list of (layer, expert) pairs, least recent first."""

    def __init__(self, S):
        self.S = S
        self.where = {}
        self.order = []

    def step(self, pairs):
        U = sorted(set(pairs), key=lambda p: (p[0], p[1]))
        hits = [p for p in U if p in self.where]
        misses = [p for p in U if p not in self.where]
        out = []
        for p in hits:
            self.order.remove(p)
            self.order.append(p)
            out.append((p, self.where[p], True, None))
        for p in misses:
            used = set(self.where.values())
            free = [s for s in range(self.S) if s not in used]
            ev = None
            if free:
                s = free[0]
            else:
                ev = self.order.pop(0)
                s = self.where.pop(ev)
            self.where[p] = s
            self.order.append(p)
            out.append((p, s, False, ev))
        return out


@pytest.mark.parametrize("L,E,S,prefetch", [(3, 8, 5, False), (4, 6, 12, True), (2, 16, 40, True),
                                            (5, 4, 3, False)])
def test_stack_cache_matches_naive_pair_list(ns, L, E, S, prefetch):
    rng = np.random.default_rng(L * 100 + E)
    C = ostack.StackCache(L, E, S, ns.lru.SlotTable)
    N = NaivePairLRU(S)
    for t in range(12):
        for l in range(L):
            if prefetch and S >= E:
                got = C.prefetch(l)
                ref = N.step([(l, e) for e in range(E)])
                assert [(a[0], a[1], a[2]) for a in got] == [(ostack.key(p[0], p[1], E), s, h)
                                                            for p, s, h, _ in ref]
            routed = rng.choice(E, size=rng.integers(1, E + 1), replace=True)
            got = C.step(l, routed)
            ref = N.step([(l, int(e)) for e in routed])
            assert [(a[0], a[1], a[2]) for a in got] == [(ostack.key(p[0], p[1], E), s, h) for p, s, h, _ in ref]
            for a, r in zip(got, ref):
                if r[3] is not None:
                    assert a[3] == ostack.key(r[3][0], r[3][1], E)
            if prefetch:
                # the layer's own step finds every routed expert resident
                assert all(a[2] for a in got)
        eo = C.expert_of
        for p, s in N.where.items():
            assert eo[s] == ostack.key(p[0], p[1], E)


def test_overlapped_prefetch_never_evicts_the_running_layer(ns):
    # with n_slots >= 2 E, layer l + 1's prefetch (issued while layer l still
    # reads its experts) takes no slot of an expert layer l's step routed
    L, E, S = 6, 8, 16
    rng = np.random.default_rng(7)
    C = ostack.StackCache(L, E, S, ns.lru.SlotTable)
    C.prefetch(0)
    for t in range(3):
        for l in range(L):
            acc = C.step(l, rng.choice(E, size=rng.integers(1, E + 1)))
            used = {a[1] for a in acc}
            if l + 1 < L:
                pf = C.prefetch(l + 1)
                assert not ({a[1] for a in pf if not a[2]} & used)
            elif t < 2:
                C.prefetch(0)


def _dense(w, fmt):
    # the dequantiser is pinned on its own (test_oracle_formats)
    from oracle import formats
    return {m: formats.dequant(w[m].codes, w[m].scales, w[m].tscale, fmt) for m in ("gate", "up", "down")}


def test_two_layer_stack_is_the_layers_in_order(ns):
    # E = 1, k = 1: each layer is one dense SwiGLU FFN with gate 1; the stack
    # computes layer 1 on bf16(layer 0's output), written out here with loops
    spec = wl.LayerSpec(E=1, k=1, d_model=32, d_ff=32, n_slots=1)
    layers, dense = [], []
    for l in range(2):
        W_r, b = wl.router_weights(spec, 40 + l)
        layers.append(ns.layer.Layer(spec, lambda e, l=l: wl.expert_weights(spec, 40 + l, e), W_r, b))
        dense.append(_dense(wl.expert_weights(spec, 40 + l, 0), spec.fmt))
    x = wl.bf16_bits_to_f64(wl.iid_tokens(1, 3, spec.d_model)[0])
    out, ys, ins, _ = ostack.stack_forward(layers, x)

    def ffn(W, v):
        d, f = spec.d_model, spec.d_ff
        y = np.zeros(d)
        h = np.zeros(f)
        for r in range(f):
            a = sum(W["gate"][r, i] * v[i] for i in range(d))
            u = sum(W["up"][r, i] * v[i] for i in range(d))
            h[r] = a / (1.0 + np.exp(-a)) * u
        for r in range(d):
            y[r] = sum(W["down"][r, j] * h[j] for j in range(f))
        return y

    for t in range(x.shape[0]):
        y0 = ffn(dense[0], x[t])
        h0 = torch.tensor(y0, dtype=torch.float64).to(torch.float32).to(torch.bfloat16).double().numpy()
        y1 = ffn(dense[1], h0)
        assert np.allclose(ys[0][t], y0, rtol=1e-12, atol=1e-12 * np.abs(y0).max())
        assert np.allclose(ys[1][t], y1, rtol=1e-12, atol=1e-12 * np.abs(y1).max())
    # the layers do not commute on these weights, so the order is pinned
    y_swapped = ffn(dense[0], ostack.bf16_round(ffn(dense[1], x[0])))
    assert not np.allclose(y_swapped, ys[1][0], rtol=1e-3)
