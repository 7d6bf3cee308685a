"""Set-up helpers around the C ABI: build a layer from per-matrix FP4 arrays.

Packing copies each expert's codes, scales and tensor scales into the byte
layout the library reports (``moe_expert_layout_for``) inside one pinned host
pool, the source of every cache fill.  No arithmetic of the layer happens
here; ``forward`` calls ``moe_forward``.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Dict, Optional

import numpy as np
import torch

from . import capi
from .workloads import BF16, CODE_BITS, LayerSpec, Matrix, MXFP4, MXFP8, NVFP4

FMT_IDS = {MXFP4: capi.MOE_MXFP4, NVFP4: capi.MOE_NVFP4, MXFP8: capi.MOE_MXFP8, BF16: capi.MOE_BF16}


def make_desc(spec: LayerSpec, max_tokens: int, act_scale_x: float = 1.0,
              act_scale_h: float = 1.0) -> capi.moe_layer_desc:
    return capi.moe_layer_desc(
        E=spec.E, k=spec.k, d_model=spec.d_model, d_ff=spec.d_ff, n_slots=spec.n_slots,
        fmt=FMT_IDS[spec.fmt],
        has_shared=int(spec.has_shared), norm_topk=int(spec.norm_topk),
        has_bias=int(spec.has_bias), max_tokens=max_tokens,
        act_scale_x=act_scale_x, act_scale_h=act_scale_h,
        prefill_act_bits=CODE_BITS[spec.prefill_act] if spec.prefill_act else 0)


def pack_expert(layout: capi.moe_expert_layout, w: Dict[str, Matrix], out: np.ndarray) -> None:
    """Write one expert (gate, up, down) into ``out`` (uint8, layout.bytes)."""
    out[:] = 0
    for name in ("gate", "up", "down"):
        m = w[name]
        c0 = getattr(layout, name + "_codes")
        s0 = getattr(layout, name + "_scales")
        out[c0:c0 + m.codes.size] = m.codes.reshape(-1)
        out[s0:s0 + m.scales.size] = m.scales.reshape(-1)
    ts = np.array([w["gate"].tscale, w["up"].tscale, w["down"].tscale], dtype=np.float32)
    t0 = layout.tensor_scales
    out[t0:t0 + 12] = ts.view(np.uint8)


def pack_pool(layout: capi.moe_expert_layout, E: int, experts_fn) -> torch.Tensor:
    """All E experts packed back to back in pinned host memory."""
    nb = layout.bytes
    pool = torch.empty(E * nb, dtype=torch.uint8, pin_memory=True)
    view = pool.numpy()
    for e in range(E):
        pack_expert(layout, experts_fn(e), view[e * nb:(e + 1) * nb])
    return pool


class MoELayer:
    """One layer on the current CUDA device, driven through the C ABI."""

    def __init__(self, spec: LayerSpec, max_tokens: int, act_scale_x: float = 1.0,
                 act_scale_h: float = 1.0, handle: Optional[int] = None):
        """handle: a stack member's handle (owned by its stack) instead of a
        new layer."""
        self.spec = spec
        self.desc = make_desc(spec, max_tokens, act_scale_x, act_scale_h)
        # the expert layout does not depend on the slot count (a stack's may exceed E)
        ld = make_desc(dataclasses.replace(spec, n_slots=min(spec.n_slots, spec.E)), max_tokens, act_scale_x,
                       act_scale_h)
        self.layout = capi.moe_expert_layout_for(ld)
        self.owned = handle is None
        self.h = capi.moe_layer_create(self.desc) if handle is None else handle
        self.pool: Optional[torch.Tensor] = None

    def close(self) -> None:
        if self.h and self.owned:
            capi.moe_layer_destroy(self.h)
        self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def expert_bytes(self) -> int:
        return self.layout.bytes

    def set_router(self, W_r: np.ndarray, bias: Optional[np.ndarray]) -> None:
        W = np.ascontiguousarray(W_r, dtype=np.float32)
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        capi.moe_set_router(self.h, W.ctypes.data, None if b is None else b.ctypes.data)

    def load_host_pool(self, experts_fn: Callable[[int], Dict[str, Matrix]], pool=None) -> None:
        """Pack all E experts into a pinned pool and register it (or register
        ``pool``, a pool packed before for the same layout: several layers
        may share one host pool)."""
        nb = self.layout.bytes
        if pool is None:
            pool = pack_pool(self.layout, self.spec.E, experts_fn)
        self.pool = pool
        capi.moe_register_host_experts(self.h, self.pool.data_ptr(), self.pool.numel())

    def set_shared(self, w: Dict[str, Matrix]) -> None:
        buf = np.zeros(self.layout.bytes, dtype=np.uint8)
        pack_expert(self.layout, w, buf)
        capi.moe_set_shared_expert(self.h, buf.ctypes.data)

    def install(self, expert: int, slot: int, stream=None) -> None:
        capi.moe_cache_install(self.h, expert, slot, stream)

    def install_all(self) -> None:
        """Expert e into slot e (a cache that holds every expert)."""
        for e in range(self.spec.E):
            self.install(e, e)
        torch.cuda.synchronize()

    def forward(self, x, y=None, stream=None, regime: int = capi.MOE_REGIME_AUTO):
        N = x.shape[0]
        if y is None:
            y = torch.empty((N, self.spec.d_model), dtype=torch.bfloat16, device=x.device)
        info = capi.moe_forward(self.h, x, N, y, stream, regime)
        return y, info


def build_layer(spec: LayerSpec, seed: int, max_tokens: int, experts_fn=None,
                install_all: bool = False, pool=None) -> MoELayer:
    """A layer with the seeded weights of ``workloads`` (router, pool, shared);
    ``pool``: an already packed host pool of the same layer shape to share."""
    from . import workloads as wl
    L = MoELayer(spec, max_tokens)
    W_r, b = wl.router_weights(spec, seed)
    L.set_router(W_r, b)
    fn = experts_fn or (lambda e: wl.expert_weights(spec, seed, e))
    L.load_host_pool(fn, pool)
    if spec.has_shared:
        L.set_shared(wl.expert_weights(spec, seed, 0, shared=True))
    if install_all:
        L.install_all()
    return L


class MoEStack:
    """n_layers layers of one shape sharing one slot pool and one LRU table
    (spec.n_slots slots for all layers); layer l has the seeded weights of
    seed + l."""

    def __init__(self, spec: LayerSpec, n_layers: int, seed: int, max_tokens: int, pools=None):
        from . import workloads as wl
        self.spec, self.n_layers = spec, n_layers
        self.desc = make_desc(spec, max_tokens)
        self.h = capi.moe_stack_create(self.desc, n_layers)
        self.layers = []
        for l in range(n_layers):
            L = MoELayer(spec, max_tokens, handle=capi.moe_stack_layer(self.h, l))
            W_r, b = wl.router_weights(spec, seed + l)
            L.set_router(W_r, b)
            pool = pools[l] if pools is not None else None
            L.load_host_pool(lambda e, l=l: wl.expert_weights(spec, seed + l, e), pool)
            if spec.has_shared:
                L.set_shared(wl.expert_weights(spec, seed + l, 0, shared=True))
            self.layers.append(L)

    def close(self) -> None:
        if self.h:
            for L in self.layers:
                L.h = None
            capi.moe_stack_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x, y=None, stream=None, regime: int = capi.MOE_REGIME_AUTO):
        N = x.shape[0]
        if y is None:
            y = torch.empty((N, self.spec.d_model), dtype=torch.bfloat16, device=x.device)
        info = capi.moe_stack_forward(self.h, x, N, y, stream, regime)
        return y, info
