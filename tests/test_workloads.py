"""Host logic of the seeded generator and the expert packing (no GPU)."""
import numpy as np
import torch

from routed_expert_layer_gemv_gb300 import capi, layer
from routed_expert_layer_gemv_gb300 import workloads as wl


def test_substreams_are_reproducible_and_independent():
    s = wl.DECODE_35B.layer
    a = wl.expert_weights(s, 0, 5)
    b = wl.expert_weights(s, 0, 5)
    c = wl.expert_weights(s, 0, 6)
    assert np.array_equal(a["gate"].codes, b["gate"].codes)
    assert not np.array_equal(a["gate"].codes, c["gate"].codes)
    assert a["gate"].codes.shape == (768, 1024) and a["down"].scales.shape == (2048, 24)


def test_weight_value_ranges():
    s = wl.DECODE_35B.layer
    w = wl.expert_weights(s, 0, 1)
    assert w["up"].scales.min() >= 119 and w["up"].scales.max() <= 123
    nv = wl.PREFILL_753B.layer
    w = wl.expert_weights(nv, 0, 1)
    e = (w["gate"].scales >> 3) & 15
    assert e.min() >= 4 and e.max() <= 8 and (w["gate"].scales < 0x80).all()
    assert w["gate"].tscale == np.float32(2 ** -6)


def test_bf16_rounding_matches_torch_via_fp32():
    x = np.random.default_rng(0).standard_normal(10000)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wl.f64_to_bf16_bits(x), ref)


def test_ar1_has_unit_variance_and_correlation():
    x, _ = wl.ar1_tokens(3, 4, 400, 256)
    v = wl.bf16_bits_to_f64(x)
    assert abs(v.var() - 1) < 0.05
    c = np.mean(v[1:] * v[:-1])
    assert abs(c - 0.9) < 0.05


def test_reject_redraws_rows():
    calls = []

    def reject(X):
        calls.append(len(X))
        return np.arange(len(X)) == 0 if len(X) > 1 else np.zeros(len(X), bool)

    x, n = wl.iid_tokens(1, 5, 128, reject)
    x0, _ = wl.iid_tokens(1, 5, 128)
    assert n == 1 and not np.array_equal(x[0], x0[0]) and np.array_equal(x[1:], x0[1:])


def test_pack_expert_places_sections():
    s = wl.TINY.layer
    d = layer.make_desc(s, 8)
    lay = capi.moe_expert_layout()
    assert capi.lib().moe_expert_layout_for(d, lay) == 0
    w = wl.expert_weights(s, 0, 3)
    buf = np.zeros(lay.bytes, np.uint8)
    layer.pack_expert(lay, w, buf)
    assert np.array_equal(buf[lay.up_codes:lay.up_codes + w["up"].codes.size], w["up"].codes.reshape(-1))
    assert np.array_equal(buf[lay.down_scales:lay.down_scales + w["down"].scales.size],
                          w["down"].scales.reshape(-1))
    ts = buf[lay.tensor_scales:lay.tensor_scales + 12].view(np.float32)
    assert list(ts) == [1.0, 1.0, 1.0]
