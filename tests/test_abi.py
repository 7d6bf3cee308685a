"""The C-ABI library builds, loads and exports every function include/moe.h
declares; the binding covers them all; host-only calls work without a GPU."""
import os
import re
import subprocess

import pytest

from routed_expert_layer_gemv_gb300 import build, capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def libpath():
    if not os.path.exists(build.lib_path()):
        build.build()
    return build.lib_path()


def test_header_declares_the_entry_points():
    names = declared()
    for must in ("moe_layer_create", "moe_cache_install", "moe_forward", "moe_lru_touch"):
        assert must in names


def test_library_exports_every_declared_symbol(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True,
                         text=True, check=True).stdout
    exported = set(l.split()[-1] for l in out.splitlines() if l.strip())
    missing = [n for n in declared() if n not in exported]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(libpath):
    assert sorted(capi.exported_symbols()) == declared()
    L = capi.lib()
    for n in declared():
        assert hasattr(L, n)


def test_status_strings_and_layout_without_gpu(libpath):
    assert capi.lib().moe_status_string(capi.MOE_ERR_ARG) == b"invalid argument"
    d = capi.moe_layer_desc(E=128, k=8, d_model=2048, d_ff=768, n_slots=47, fmt=capi.MOE_MXFP4,
                            has_shared=0, norm_topk=1, has_bias=0, max_tokens=16,
                            act_scale_x=1.0, act_scale_h=1.0)
    lay = capi.moe_expert_layout_for(d)
    # 3 matrices of 768 x 2048 FP4 codes + E8M0 scales per 32, 256-byte aligned
    assert lay.gate_codes == 0 and lay.up_codes == 768 * 1024
    assert lay.gate_scales == 3 * 768 * 1024
    assert lay.tensor_scales == 3 * 768 * 1024 + 3 * 768 * 64
    assert lay.bytes == lay.tensor_scales + 256
    for off in (lay.up_codes, lay.down_codes, lay.gate_scales, lay.up_scales, lay.down_scales):
        assert off % 256 == 0


@pytest.mark.parametrize("field,value", [("E", 0), ("k", 0), ("k", 129), ("d_model", 100),
                                         ("d_ff", 0), ("n_slots", 0), ("n_slots", 129),
                                         ("fmt", 7), ("max_tokens", 0)])
def test_invalid_descriptor_rejected_without_gpu(libpath, field, value):
    d = capi.moe_layer_desc(E=128, k=8, d_model=2048, d_ff=768, n_slots=47, fmt=capi.MOE_MXFP4,
                            has_shared=0, norm_topk=1, has_bias=0, max_tokens=16,
                            act_scale_x=1.0, act_scale_h=1.0)
    setattr(d, field, value)
    out = capi.moe_expert_layout()
    assert capi.lib().moe_expert_layout_for(d, out) == capi.MOE_ERR_ARG


@pytest.mark.parametrize("fmt,bits,ok", [(capi.MOE_MXFP4, 0, True), (capi.MOE_MXFP4, 4, True),
                                         (capi.MOE_MXFP4, 8, True), (capi.MOE_NVFP4, 8, False),
                                         (capi.MOE_NVFP4, 4, True), (capi.MOE_MXFP8, 8, True),
                                         (capi.MOE_MXFP8, 4, False), (capi.MOE_BF16, 8, False),
                                         (capi.MOE_BF16, 16, True), (capi.MOE_MXFP4, 16, False)])
def test_prefill_activation_format_checked_without_gpu(libpath, fmt, bits, ok):
    # W4A8 (MXFP8 activations) exists for MXFP4 weights only: NVFP4's E4M3
    # scales per 16 have no kind::mxf8f6f4 block-scale form
    d = capi.moe_layer_desc(E=8, k=2, d_model=256, d_ff=512, n_slots=8, fmt=fmt,
                            has_shared=0, norm_topk=1, has_bias=0, max_tokens=16,
                            act_scale_x=1.0, act_scale_h=1.0, prefill_act_bits=bits)
    out = capi.moe_expert_layout()
    assert capi.lib().moe_expert_layout_for(d, out) == (capi.MOE_OK if ok else capi.MOE_ERR_ARG)


def test_nvfp4_scales_must_be_powers_of_two(libpath):
    d = capi.moe_layer_desc(E=8, k=2, d_model=256, d_ff=512, n_slots=8, fmt=capi.MOE_NVFP4,
                            has_shared=0, norm_topk=1, has_bias=0, max_tokens=16,
                            act_scale_x=0.75, act_scale_h=1.0)
    out = capi.moe_expert_layout()
    assert capi.lib().moe_expert_layout_for(d, out) == capi.MOE_ERR_ARG
    d.act_scale_x = 0.5
    assert capi.lib().moe_expert_layout_for(d, out) == capi.MOE_OK
