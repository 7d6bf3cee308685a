"""Shared test helpers: seeded layers on both sides, the output tolerance."""
from __future__ import annotations

import dataclasses
from collections import OrderedDict

import numpy as np
import pytest
import torch

from oracle.native import layer as olayer
from routed_expert_layer_gemv_gb300 import workloads as wl

# Output tolerance of the layer (bf16 activations, fp32 accumulation):
# relative Frobenius error <= 5e-3 and per-element |err| <= 3e-2 * RMS(ref).
REL_FRO = 5e-3
MAX_ABS_RMS = 3e-2


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def assert_close_layer(y_gpu, y_ref, what=""):
    y = y_gpu.float().cpu().double().numpy() if isinstance(y_gpu, torch.Tensor) else np.asarray(y_gpu, np.float64)
    ref = np.asarray(y_ref, np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    err = y - ref
    rms = np.sqrt(np.mean(ref * ref))
    fro = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    mx = np.abs(err).max() if err.size else 0.0
    assert fro <= REL_FRO, "%s rel Frobenius %.3e > %.1e" % (what, fro, REL_FRO)
    assert mx <= MAX_ABS_RMS * rms, "%s max |err| %.3e > %.1e * RMS %.3e" % (what, mx, MAX_ABS_RMS, rms)
    return fro, mx / max(rms, 1e-300)


class CachedExperts:
    """Generator weights per expert, memoised (bounded)."""

    def __init__(self, spec, seed, cap=64):
        self.spec, self.seed, self.cap = spec, seed, cap
        self.cache = OrderedDict()

    def __call__(self, e):
        if e in self.cache:
            self.cache.move_to_end(e)
            return self.cache[e]
        w = wl.expert_weights(self.spec, self.seed, e)
        self.cache[e] = w
        if len(self.cache) > self.cap:
            self.cache.popitem(last=False)
        return w


def oracle_layer(spec, seed, experts=None):
    W_r, b = wl.router_weights(spec, seed)
    sh = wl.expert_weights(spec, seed, 0, shared=True) if spec.has_shared else None
    return olayer.Layer(spec, experts or CachedExperts(spec, seed), W_r, b, sh)


def reject_near_ties(spec, seed):
    W_r, b = wl.router_weights(spec, seed)
    return lambda X: olayer.near_tie(X, W_r, b, spec.k, 1e-4)


def small_spec(**kw):
    base = dict(E=8, k=2, d_model=256, d_ff=512, n_slots=8)
    base.update(kw)
    return wl.LayerSpec(**base)


def bf16_tensor(bits: np.ndarray, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device else t


def check_last_step(L, spec, N, idx_ref, gates_ref):
    """The router and permutation arrays of the layer's last moe_forward --
    the ones its expert FFN and combine used -- against the oracle: ids and
    permutation bit for bit, gates to fp32 rounding."""
    from routed_expert_layer_gemv_gb300 import capi
    k, E = spec.k, spec.E
    i32 = dict(dtype=torch.int32, device="cuda")
    idx = torch.full((N * k,), -7, **i32)
    gates = torch.full((N * k,), -7.0, dtype=torch.float32, device="cuda")
    counts, offsets = torch.full((E,), -7, **i32), torch.full((E + 1,), -7, **i32)
    row_of, tok_of = torch.full((N * k,), -7, **i32), torch.full((N * k,), -7, **i32)
    n = capi.moe_debug_last_step(L.h, idx, gates, counts, offsets, row_of, tok_of)
    torch.cuda.synchronize()
    assert n == N
    idx_ref = np.asarray(idx_ref).reshape(N, k)
    assert np.array_equal(idx.cpu().numpy().reshape(N, k), idx_ref)
    rc, ro, rr, rt = olayer.permute(idx_ref, E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(row_of.cpu().numpy(), rr.reshape(-1))
    assert np.array_equal(tok_of.cpu().numpy(), rt)
    assert np.allclose(gates.cpu().numpy().reshape(N, k), gates_ref, rtol=2e-6, atol=1e-7)
