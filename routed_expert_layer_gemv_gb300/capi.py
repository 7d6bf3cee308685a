"""ctypes binding of the layer's C ABI (include/moe.h).

Argument marshalling only: every step of the forward pass runs in the CUDA
library.  If ``libmoe_gb300.so`` has not been built, importing the binding
still works but the first call raises ``RuntimeError`` -- there is no
fallback of any kind.

Functions keep the C names (``moe_layer_create`` ...).  Pointers are passed
as Python ints (``tensor.data_ptr()``), ``ctypes`` arrays or ``None``.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

from . import build as _build

MOE_OK = 0
MOE_ERR_ARG = -1
MOE_ERR_NOT_INSTALLED = -2
MOE_ERR_OOM = -3
MOE_ERR_FILL = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_CUDA = -6
MOE_ERR_STATE = -7
MOE_ERR_UNSUPPORTED = -8

MOE_MXFP4 = 0
MOE_NVFP4 = 1
MOE_MXFP8 = 2
MOE_BF16 = 3

MOE_PROF_NAMES = ["router", "permute", "lru", "gateup", "down", "combine", "fill", "prefill", "commit",
                  "step"]

MOE_DECODE_AUTO = 0
MOE_DECODE_CHAIN = 1
MOE_DECODE_STEP = 2

MOE_FILL_MEMCPY = 0
MOE_FILL_DEVICE = 1
MOE_FILL_KERNEL = 2
MOE_FILL_FUSED = 3
MOE_FILL_AUTO = 4

MOE_INJECT_NONE = 0
MOE_INJECT_FILL = 1
MOE_INJECT_WAIT_LIMIT = 2

MOE_REGIME_AUTO = 0
MOE_REGIME_DECODE = 1
MOE_REGIME_PREFILL = 2

MOE_PREFETCH_AUTO = 0
MOE_PREFETCH_NONE = 1
MOE_PREFETCH_SERIAL = 2
MOE_PREFETCH_OVERLAP = 3


class moe_layer_desc(C.Structure):
    _fields_ = [("E", C.c_int), ("k", C.c_int), ("d_model", C.c_int), ("d_ff", C.c_int),
                ("n_slots", C.c_int), ("fmt", C.c_int), ("has_shared", C.c_int),
                ("norm_topk", C.c_int), ("has_bias", C.c_int), ("max_tokens", C.c_int),
                ("act_scale_x", C.c_float), ("act_scale_h", C.c_float), ("prefill_act_bits", C.c_int)]


class moe_expert_layout(C.Structure):
    _fields_ = [("bytes", C.c_size_t), ("gate_codes", C.c_size_t), ("up_codes", C.c_size_t),
                ("down_codes", C.c_size_t), ("gate_scales", C.c_size_t),
                ("up_scales", C.c_size_t), ("down_scales", C.c_size_t),
                ("tensor_scales", C.c_size_t)]


class moe_forward_info(C.Structure):
    _fields_ = [("regime", C.c_int), ("n_tokens", C.c_int), ("n_distinct", C.c_int),
                ("n_hits", C.c_int), ("n_misses", C.c_int), ("n_waves", C.c_int),
                ("fill_bytes", C.c_size_t), ("host_synced", C.c_int), ("n_launches", C.c_int),
                ("fused_step", C.c_int)]


_P = C.c_void_p
_I = C.c_int
_SIGS = {
    "moe_expert_layout_for": ([C.POINTER(moe_layer_desc), C.POINTER(moe_expert_layout)], _I),
    "moe_layer_create": ([C.POINTER(moe_layer_desc), C.POINTER(_P)], _I),
    "moe_layer_destroy": ([_P], _I),
    "moe_set_router": ([_P, _P, _P], _I),
    "moe_register_host_experts": ([_P, _P, C.c_size_t], _I),
    "moe_set_shared_expert": ([_P, _P], _I),
    "moe_cache_install": ([_P, _I, _I, _P], _I),
    "moe_cache_resize": ([_P, _I, _P], _I),
    "moe_lru_touch": ([_P, _P, _I, _P, _P, _P, _P, _P], _I),
    "moe_lru_get_state": ([_P, _P, _P, _P], _I),
    "moe_lru_set_state": ([_P, _P, _P, C.c_uint64], _I),
    "moe_forward": ([_P, _P, _I, _P, _P, _I, C.POINTER(moe_forward_info)], _I),
    "moe_set_fill_mode": ([_P, _I], _I),
    "moe_set_decode_path": ([_P, _I], _I),
    "moe_stats": ([_P, _P], _I),
    "moe_profile": ([_P, _I], _I),
    "moe_profile_read": ([_P, _P, _P], _I),
    "moe_last_error": ([_P], C.c_char_p),
    "moe_status_string": ([_I], C.c_char_p),
    "moe_debug_router": ([_P, _P, _I, _P, _P, _P, _P], _I),
    "moe_debug_permute": ([_P, _P, _I, _P, _P, _P, _P, _P], _I),
    "moe_debug_last_step": ([_P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_debug_last_hidden": ([_P, _P, _P, _P, _P], _I),
    "moe_debug_inject": ([_P, _I, C.c_longlong], _I),
    "moe_debug_alloc_fault": ([C.c_longlong, _P], _I),
    "moe_debug_step_trace": ([_P, _P, _I, _P, _P], _I),
    "moe_debug_dequant": ([_P, _I, _I, _P, _P], _I),
    "moe_debug_actquant": ([_P, _P, _I, _I, _P, _P, _I, _P], _I),
    "moe_permute_noalloc": ([_P, _I, _I, _I, _P, _P, _P, _P, _P, C.c_char_p, C.c_size_t], _I),
    "moe_stack_create": ([C.POINTER(moe_layer_desc), _I, C.POINTER(_P)], _I),
    "moe_stack_destroy": ([_P], _I),
    "moe_stack_layer": ([_P, _I, C.POINTER(_P)], _I),
    "moe_stack_set_prefetch": ([_P, _I], _I),
    "moe_stack_set_prefetch_copy": ([_P, _I], _I),
    "moe_stack_forward": ([_P, _P, _I, _P, _P, _I, C.POINTER(moe_forward_info)], _I),
    "moe_stack_prefetch_stats": ([_P, _P], _I),
    "moe_stack_last_error": ([_P], C.c_char_p),
}

_lib: Optional[C.CDLL] = None


def library_path() -> str:
    return _build.lib_path()


def lib() -> C.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                "libmoe_gb300.so is not built (expected at %s); run "
                "`python -m routed_expert_layer_gemv_gb300.build`" % path)
        L = C.CDLL(path)
        for name, (argt, rest) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = argt
            fn.restype = rest
        _lib = L
    return _lib


def exported_symbols():
    return sorted(_SIGS)


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s (%d): %s" % (lib().moe_status_string(status).decode(), status, msg))
        self.status = status


def check(status: int, handle=None) -> None:
    if status != MOE_OK:
        msg = lib().moe_last_error(handle).decode() if handle else ""
        raise MoeError(status, msg)


def check_stack(status: int, stack) -> None:
    if status != MOE_OK:
        raise MoeError(status, lib().moe_stack_last_error(stack).decode() if stack else "")


def _ptr(p) -> Optional[int]:
    if p is None:
        return None
    if isinstance(p, int):
        return p
    if hasattr(p, "data_ptr"):
        return p.data_ptr()
    return C.cast(p, C.c_void_p).value


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ---- thin wrappers with the C names ------------------------------------

def moe_expert_layout_for(desc: moe_layer_desc) -> moe_expert_layout:
    out = moe_expert_layout()
    check(lib().moe_expert_layout_for(C.byref(desc), C.byref(out)))
    return out


def moe_layer_create(desc: moe_layer_desc) -> int:
    h = C.c_void_p()
    rc = lib().moe_layer_create(C.byref(desc), C.byref(h))
    check(rc)
    return h.value


def moe_layer_destroy(h: int) -> None:
    check(lib().moe_layer_destroy(h))


def moe_set_router(h, W_r, bias=None) -> None:
    check(lib().moe_set_router(h, _ptr(W_r), _ptr(bias)), h)


def moe_register_host_experts(h, pool, nbytes: int) -> None:
    check(lib().moe_register_host_experts(h, _ptr(pool), nbytes), h)


def moe_set_shared_expert(h, weights) -> None:
    check(lib().moe_set_shared_expert(h, _ptr(weights)), h)


def moe_cache_install(h, expert: int, slot: int, stream=None) -> None:
    check(lib().moe_cache_install(h, expert, slot, _stream(stream)), h)


def moe_cache_resize(h, n_slots: int, stream=None) -> None:
    check(lib().moe_cache_resize(h, n_slots, _stream(stream)), h)


def moe_lru_touch(h, experts, stream=None):
    """Returns (slot_of per input, miss experts, miss slots)."""
    n = len(experts)
    arr = (C.c_int * max(1, n))(*experts)
    slots = (C.c_int * max(1, n))()
    me = (C.c_int * max(1, n))()
    ms = (C.c_int * max(1, n))()
    nm = C.c_int()
    check(lib().moe_lru_touch(h, arr, n, slots, me, ms, C.byref(nm), _stream(stream)), h)
    return list(slots[:n]), list(me[:nm.value]), list(ms[:nm.value])


def moe_lru_get_state(h, n_slots: int):
    eo = (C.c_int * n_slots)()
    st = (C.c_uint64 * n_slots)()
    clk = C.c_uint64()
    check(lib().moe_lru_get_state(h, eo, st, C.byref(clk)), h)
    return list(eo), list(st), clk.value


def moe_lru_set_state(h, expert_of_slot, stamps, clock: int) -> None:
    n = len(expert_of_slot)
    eo = (C.c_int * n)(*expert_of_slot)
    st = (C.c_uint64 * n)(*stamps)
    check(lib().moe_lru_set_state(h, eo, st, clock), h)


def moe_forward(h, x, N: int, y, stream=None, regime: int = MOE_REGIME_AUTO) -> moe_forward_info:
    info = moe_forward_info()
    check(lib().moe_forward(h, _ptr(x), N, _ptr(y), _stream(stream), regime, C.byref(info)), h)
    return info


def moe_set_fill_mode(h, mode: int) -> None:
    check(lib().moe_set_fill_mode(h, mode), h)


def moe_set_decode_path(h, path: int) -> None:
    check(lib().moe_set_decode_path(h, path), h)


def moe_stats(h):
    """(steps, distinct experts, hits, misses) accumulated on the device."""
    out = (C.c_uint64 * 4)()
    check(lib().moe_stats(h, out), h)
    return tuple(out)


def moe_profile(h, enable: bool) -> None:
    check(lib().moe_profile(h, int(enable)), h)


def moe_profile_read(h):
    """{class name: (device ms summed, launches)}."""
    n = len(MOE_PROF_NAMES)
    ms = (C.c_double * n)()
    cnt = (C.c_int * n)()
    check(lib().moe_profile_read(h, ms, cnt), h)
    return {name: (ms[i], cnt[i]) for i, name in enumerate(MOE_PROF_NAMES)}


def moe_debug_router(h, x, N, idx, gates, logits=None, stream=None) -> None:
    check(lib().moe_debug_router(h, _ptr(x), N, _ptr(idx), _ptr(gates), _ptr(logits),
                                 _stream(stream)), h)


def moe_debug_permute(h, idx, N, counts, offsets, row_of, tok_of, stream=None) -> None:
    check(lib().moe_debug_permute(h, _ptr(idx), N, _ptr(counts), _ptr(offsets), _ptr(row_of),
                                  _ptr(tok_of), _stream(stream)), h)


def moe_debug_last_step(h, idx=None, gates=None, counts=None, offsets=None, row_of=None,
                        tok_of=None, stream=None) -> int:
    """Copies the last moe_forward's router and permutation arrays into the
    given device tensors; returns that call's token count."""
    n = C.c_int(0)
    check(lib().moe_debug_last_step(h, _ptr(idx), _ptr(gates), _ptr(counts), _ptr(offsets),
                                    _ptr(row_of), _ptr(tok_of), C.byref(n), _stream(stream)), h)
    return n.value


def moe_debug_last_hidden(h, hidden=None, hq_codes=None, hq_scales=None, stream=None) -> None:
    check(lib().moe_debug_last_hidden(h, _ptr(hidden), _ptr(hq_codes), _ptr(hq_scales),
                                      _stream(stream)), h)


def moe_debug_inject(h, what: int, arg: int = 0) -> None:
    check(lib().moe_debug_inject(h, what, arg), h)


def moe_debug_alloc_fault(nth: int):
    """Arms the allocation fault (0 disarms); returns the live (device, pinned) allocation counts."""
    live = (C.c_longlong * 2)()
    check(lib().moe_debug_alloc_fault(nth, live))
    return live[0], live[1]


def moe_debug_step_trace(h):
    """Per-CTA global-timer marks (ns) of the last fused step run under
    moe_profile, as a list of rows (one per CTA)."""
    G, M = C.c_int(0), C.c_int(0)
    lib().moe_debug_step_trace(h, None, 0, C.byref(G), C.byref(M))
    buf = (C.c_uint64 * max(1, G.value * M.value))()
    check(lib().moe_debug_step_trace(h, buf, G.value * M.value, None, None), h)
    return [list(buf[c * M.value:(c + 1) * M.value]) for c in range(G.value)]


def moe_debug_dequant(h, slot: int, m: int, out, stream=None) -> None:
    check(lib().moe_debug_dequant(h, slot, m, _ptr(out), _stream(stream)), h)


def moe_debug_actquant(h, v, rows: int, K: int, codes, scales, which: int = 0, stream=None) -> None:
    check(lib().moe_debug_actquant(h, _ptr(v), rows, K, _ptr(codes), _ptr(scales), which,
                                   _stream(stream)), h)


def moe_permute_noalloc(idx, N: int, k: int, E: int, counts, offsets, row_of, tok_of,
                        stream=None) -> None:
    """The permutation without a layer handle and without allocating (see moe.h)."""
    err = C.create_string_buffer(256)
    rc = lib().moe_permute_noalloc(_ptr(idx), N, k, E, _ptr(counts), _ptr(offsets),
                                   _ptr(row_of), _ptr(tok_of), _stream(stream), err, len(err))
    if rc != MOE_OK:
        raise MoeError(rc, err.value.decode())


# ---- stacks --------------------------------------------------------------

def moe_stack_create(desc: moe_layer_desc, n_layers: int) -> int:
    h = C.c_void_p()
    check(lib().moe_stack_create(C.byref(desc), n_layers, C.byref(h)))
    return h.value


def moe_stack_destroy(s: int) -> None:
    check(lib().moe_stack_destroy(s))


def moe_stack_layer(s: int, l: int) -> int:
    h = C.c_void_p()
    check_stack(lib().moe_stack_layer(s, l, C.byref(h)), s)
    return h.value


def moe_stack_set_prefetch(s: int, mode: int) -> None:
    check_stack(lib().moe_stack_set_prefetch(s, mode), s)


def moe_stack_set_prefetch_copy(s: int, fill: int) -> None:
    check_stack(lib().moe_stack_set_prefetch_copy(s, fill), s)


def moe_stack_forward(s, x, N: int, y, stream=None, regime: int = MOE_REGIME_AUTO) -> moe_forward_info:
    info = moe_forward_info()
    check_stack(lib().moe_stack_forward(s, _ptr(x), N, _ptr(y), _stream(stream), regime, C.byref(info)), s)
    return info


def moe_stack_prefetch_stats(s):
    """(prefetch steps, keys accessed, hits, misses) accumulated on the device."""
    out = (C.c_uint64 * 4)()
    check_stack(lib().moe_stack_prefetch_stats(s, out), s)
    return tuple(out)
