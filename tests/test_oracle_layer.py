"""Pins of the oracle's router, permutation, SwiGLU experts and combine
against brute force, textbook loops, library routines and invariants (no GPU)."""
import dataclasses
import math

import numpy as np
import pytest

from conftest import ORACLES, swap_oracle
import scipy.special

from oracle import formats, layer
from routed_expert_layer_gemv_gb300 import workloads as wl


@pytest.fixture(autouse=True, params=ORACLES)
def oracle_impl(request, monkeypatch):
    return swap_oracle(__name__, request, monkeypatch, ("formats", "layer"))



# ---------------------------------------------------------------- router

def _brute_topk(L, k):
    out = []
    for row in L:
        order = sorted(range(len(row)), key=lambda e: (-row[e], e))
        out.append(sorted(order[:k]))
    return np.array(out)


def test_topk_vs_brute_force_with_ties_and_bias():
    g = np.random.default_rng(1)
    N, d, E, k = 40, 16, 12, 4
    x = np.round(g.standard_normal((N, d)) * 4) / 4
    W = np.round(g.standard_normal((E, d)) * 2) / 2
    W[5] = W[2]            # exact ties: expert 2 must win over 5
    W[9] = W[0]
    b = np.zeros(E)
    b[7] = 0.5
    idx, gates, L = layer.router(x, W, b, k)
    Lb = np.array([[sum(x[t, i] * W[e, i] for i in range(d)) + b[e] for e in range(E)] for t in range(N)])
    assert np.allclose(L, Lb, rtol=0, atol=1e-12)
    assert np.array_equal(idx, _brute_topk(Lb, k))


def test_equal_logits_give_uniform_gates_and_lowest_ids():
    N, d, E = 3, 8, 6
    x = np.ones((N, d))
    idx, gates, _ = layer.router(x, np.zeros((E, d)), None, E)
    assert np.array_equal(idx, np.tile(np.arange(E), (N, 1)))
    assert np.allclose(gates, 1.0 / E, rtol=0, atol=1e-15)
    idx2, _, _ = layer.router(x, np.zeros((E, d)), None, 2)
    assert np.array_equal(idx2, np.tile([0, 1], (N, 1)))


def test_gates_renormalised_and_full_softmax():
    g = np.random.default_rng(2)
    x, W = g.standard_normal((20, 32)), g.standard_normal((10, 32)) / 5
    idx, gates, L = layer.router(x, W, None, 3, norm_topk=True)
    assert np.allclose(gates.sum(1), 1.0)
    p = scipy.special.softmax(L, axis=1)
    sel = np.take_along_axis(p, idx, 1)
    assert np.allclose(gates, sel / sel.sum(1, keepdims=True))
    _, gates0, _ = layer.router(x, W, None, 3, norm_topk=False)
    assert np.allclose(gates0, sel)


def test_near_tie_vs_brute_force():
    g = np.random.default_rng(3)
    x, W = g.standard_normal((200, 8)), g.standard_normal((16, 8))
    k = 5
    L = x @ W.T
    want = []
    for row in L:
        s = sorted(row, reverse=True)
        want.append(s[k - 1] - s[k] < 0.05)
    assert np.array_equal(layer.near_tie(x, W, None, k, 0.05), np.array(want))


# ---------------------------------------------------------------- permute

def test_permute_definitions():
    g = np.random.default_rng(4)
    N, E, k = 37, 9, 3
    idx = np.sort(np.array([g.choice(E, k, replace=False) for _ in range(N)]), 1)
    counts, offsets, row_of, tok_of = layer.permute(idx, E)
    assert counts.sum() == N * k
    for e in range(E):
        assert counts[e] == sum(int(e in idx[t]) for t in range(N))
        assert offsets[e] == sum(counts[:e])
    for t in range(N):
        for j in range(k):
            e = idx[t, j]
            # rank among earlier tokens routed to e
            rank = sum(1 for t2 in range(t) if e in idx[t2])
            assert row_of[t, j] == offsets[e] + rank
            assert tok_of[row_of[t, j]] == t
    assert sorted(row_of.reshape(-1)) == list(range(N * k))


# ---------------------------------------------------------------- experts

def _tiny_spec(fmt="mxfp4", E=1, k=1, d=64, f=32, shared=False):
    return wl.LayerSpec(E=E, k=k, d_model=d, d_ff=f, n_slots=E, fmt=fmt, has_shared=shared)


def _swiglu_loops(xrow, Wg, Wu, Wd):
    f, d = Wg.shape
    h = []
    for r in range(f):
        a = sum(Wg[r, i] * xrow[i] for i in range(d))
        u = sum(Wu[r, i] * xrow[i] for i in range(d))
        h.append(a / (1.0 + math.exp(-a)) * u)
    return np.array([sum(Wd[c, r] * h[r] for r in range(f)) for c in range(d)])


def test_silu_vs_scipy():
    z = np.linspace(-30, 30, 301)
    assert np.allclose(layer.silu(z), z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_single_expert_layer_is_dense_swiglu(fmt):
    spec = _tiny_spec(fmt)
    w = wl.expert_weights(spec, 11, 0)
    W_r, _ = wl.router_weights(spec, 11)
    L = layer.Layer(spec, lambda e: w, W_r, None)
    x = wl.bf16_bits_to_f64(wl.iid_tokens(11, 5, spec.d_model)[0])
    y, idx, gates = L.forward(x)
    assert (idx == 0).all() and np.allclose(gates, 1.0)
    Wd = {n: formats.dequant(m.codes, m.scales, m.tscale, fmt) for n, m in w.items()}
    for t in range(5):
        ref = _swiglu_loops(x[t], Wd["gate"], Wd["up"], Wd["down"])
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-12)


def _layer(spec, seed=5):
    W_r, b = wl.router_weights(spec, seed)
    ex = {e: wl.expert_weights(spec, seed, e) for e in range(spec.E)}
    sh = wl.expert_weights(spec, seed, 0, shared=True) if spec.has_shared else None
    return layer.Layer(spec, lambda e: ex[e], W_r, b, sh)


def test_zero_input_gives_zero_output():
    spec = _tiny_spec(E=4, k=2, shared=True)
    L = _layer(spec)
    for regime in ("decode", "prefill"):
        y, _, _ = L.forward(np.zeros((3, spec.d_model)), regime)
        assert not y.any()


def test_k_equals_E_with_equal_gates_is_expert_mean():
    spec = _tiny_spec(E=3, k=3)
    L = _layer(spec)
    L.W_r = np.zeros_like(L.W_r)
    x = wl.bf16_bits_to_f64(wl.iid_tokens(6, 4, spec.d_model)[0])
    y, _, gates = L.forward(x)
    assert np.allclose(gates, 1 / 3)
    ref = np.zeros_like(y)
    for e in range(3):
        W = L.expert(e)
        ref += np.array([_swiglu_loops(x[t], W["gate"], W["up"], W["down"]) for t in range(4)]) / 3
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_token_permutation_invariance():
    spec = _tiny_spec(E=6, k=2, shared=True)
    L = _layer(spec)
    x = wl.bf16_bits_to_f64(wl.iid_tokens(7, 10, spec.d_model)[0])
    perm = np.random.default_rng(0).permutation(10)
    for regime in ("decode", "prefill"):
        y, _, _ = L.forward(x, regime)
        yp, _, _ = L.forward(x[perm], regime)
        # FP64 with BLAS: equal up to the last bits of a blocked matmul
        assert np.allclose(yp, y[perm], rtol=1e-12, atol=1e-14)
        ys, _, _ = L.forward(x, regime, tokens=[3, 7])
        assert np.allclose(ys, y[[3, 7]], rtol=1e-12, atol=1e-14)


def test_combine_linear_in_gates_and_shared_added():
    g = np.random.default_rng(12)
    O = g.standard_normal((12, 5))
    row_of = np.arange(12).reshape(4, 3)
    g1, g2 = g.standard_normal((4, 3)), g.standard_normal((4, 3))
    s = g.standard_normal((4, 5))
    c = layer.combine
    assert np.allclose(c(O, g1 + g2, row_of), c(O, g1, row_of) + c(O, g2, row_of))
    assert np.allclose(c(O, g1, row_of, s) - c(O, g1, row_of), s)
    want = np.array([[sum(g1[t, j] * O[row_of[t, j], i] for j in range(3)) for i in range(5)] for t in range(4)])
    assert np.allclose(c(O, g1, row_of), want)


def test_shared_expert_is_added_with_weight_one():
    spec = _tiny_spec(E=4, k=2, shared=True)
    L = _layer(spec)
    x = wl.bf16_bits_to_f64(wl.iid_tokens(9, 3, spec.d_model)[0])
    y, _, _ = L.forward(x)
    L2 = _layer(spec)
    L2.spec = _tiny_spec(E=4, k=2, shared=False)
    y0, _, _ = L2.forward(x)
    Ws = layer.dequant_expert(L.shared_w, spec.fmt)
    s = np.array([_swiglu_loops(x[t], Ws["gate"], Ws["up"], Ws["down"]) for t in range(3)])
    assert np.allclose(y - y0, s, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_prefill_regime_is_decode_on_quantised_activations(fmt):
    spec = _tiny_spec(fmt)
    w = wl.expert_weights(spec, 13, 0)
    W = layer.dequant_expert(w, fmt)
    x = wl.bf16_bits_to_f64(wl.iid_tokens(13, 4, spec.d_model)[0])
    xq = layer.act_roundtrip(x, fmt, 1.0)
    for t in range(4):
        a = W["gate"] @ xq[t]
        u = W["up"] @ xq[t]
        h = layer.act_roundtrip((a / (1 + np.exp(-a)) * u)[None, :], fmt, 1.0)[0]
        assert np.allclose(layer.expert_ffn(x[t:t + 1], W, "prefill", fmt)[0], W["down"] @ h,
                           rtol=1e-12, atol=1e-12)
    # quantised x differs from x, but not by more than the FP4 grid allows
    assert not np.array_equal(xq, x)
    assert np.abs(xq - x).max() <= np.abs(x).max() / 3


def test_w4a8_prefill_is_dense_swiglu_on_mxfp8_activations():
    # MXFP4 weights with MXFP8 activations: x and h rounded by the MXFP8
    # quantiser (pinned on its own in test_oracle_quant), the FFN written out
    # with loops; the result is not the W4A4 one
    from oracle import quant
    spec = wl.LayerSpec(E=1, k=1, d_model=64, d_ff=64, n_slots=1, prefill_act=wl.MXFP8)
    w = wl.expert_weights(spec, 17, 0)
    W_r, _ = wl.router_weights(spec, 17)
    L = layer.Layer(spec, lambda e: w, W_r, None)
    x = wl.bf16_bits_to_f64(wl.iid_tokens(17, 4, spec.d_model)[0])
    y, _, _ = L.forward(x, "prefill")
    Wd = {n: formats.dequant(m.codes, m.scales, m.tscale, "mxfp4") for n, m in w.items()}

    def rt8(v):
        c, s = quant.quant_mxfp8(np.asarray(v, np.float64)[None, :])
        return formats.dequant(c, s, 1.0, "mxfp8")[0]

    for t in range(4):
        xq = rt8(x[t])
        f = spec.d_ff
        h = np.zeros(f)
        for r in range(f):
            a = sum(Wd["gate"][r, i] * xq[i] for i in range(spec.d_model))
            u = sum(Wd["up"][r, i] * xq[i] for i in range(spec.d_model))
            h[r] = a / (1.0 + math.exp(-a)) * u
        hq = rt8(h)
        ref = np.array([sum(Wd["down"][r, j] * hq[j] for j in range(f)) for r in range(spec.d_model)])
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    L4 = layer.Layer(dataclasses.replace(spec, prefill_act=None), lambda e: w, W_r, None)
    y4, _, _ = L4.forward(x, "prefill")
    assert not np.allclose(y, y4, rtol=1e-3)


def test_native_and_numpy_oracles_agree():
    # the two implementations of the oracle, on layers with every option:
    # ids, permutation and quantiser codes exactly, values to FP64 rounding
    from oracle import layer as np_layer
    from oracle.native import layer as cpp_layer
    for fmt, shared, bias, act in (("mxfp4", False, False, None), ("nvfp4", True, True, None),
                                   ("mxfp8", True, False, None), ("bf16", False, True, None),
                                   ("mxfp4", True, False, "mxfp8")):
        spec = wl.LayerSpec(E=12, k=3, d_model=128, d_ff=64, n_slots=12, fmt=fmt, has_shared=shared,
                            has_bias=bias, prefill_act=act)
        W_r, b = wl.router_weights(spec, 8)
        ex = {e: wl.expert_weights(spec, 8, e) for e in range(spec.E)}
        sh = wl.expert_weights(spec, 8, 0, shared=True) if shared else None
        x = wl.bf16_bits_to_f64(wl.iid_tokens(8, 17, spec.d_model)[0])
        for regime in ("decode", "prefill"):
            y1, i1, g1 = cpp_layer.Layer(spec, lambda e: ex[e], W_r, b, sh).forward(x, regime)
            y2, i2, g2 = np_layer.Layer(spec, lambda e: ex[e], W_r, b, sh).forward(x, regime)
            assert np.array_equal(i1, i2)
            assert np.allclose(g1, g2, rtol=1e-14, atol=0)
            assert np.allclose(y1, y2, rtol=1e-12, atol=1e-12 * np.abs(y2).max())
            for a, c in zip(cpp_layer.permute(i1, spec.E), np_layer.permute(i2, spec.E)):
                assert np.array_equal(a, c)
