"""Pins of the oracle's FP4 formats against the public encodings, IEEE bit
layouts and torch's float8 conversion (no GPU)."""
import math

import numpy as np
import pytest
import torch

from conftest import ORACLES, read_golden, swap_oracle
from oracle import formats, quant


@pytest.fixture(autouse=True, params=ORACLES)
def oracle_impl(request, monkeypatch):
    return swap_oracle(__name__, request, monkeypatch, ("formats", "quant"))


def test_e2m1_table_matches_spec_fixture():
    rows = read_golden("e2m1_values.txt")
    assert len(rows) == 16
    for code, val in rows:
        got = formats.E2M1_TABLE[int(code)]
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e2m1_via_fp16_bit_placement():
    # independent route: the 3 magnitude bits placed as fp16 exponent-low/mantissa-top
    # bits give 2^(e-15)(1+m/2) (or the subnormal m*2^-15); times 2^14 is the value.
    for c in range(16):
        bits = ((c & 7) << 9) | ((c & 8) << 12)
        h = np.array([bits], dtype=np.uint16).view(np.float16)[0]
        assert float(h) * 2.0 ** 14 == formats.E2M1_TABLE[c]


def test_e8m0_is_the_fp32_exponent_field():
    for x in range(1, 255):
        f = np.array([x << 23], dtype=np.uint32).view(np.float32)[0]
        assert float(f) == formats.E8M0_TABLE[x]
    sub = np.array([0x00400000], dtype=np.uint32).view(np.float32)[0]  # 2^-127
    assert float(sub) == formats.E8M0_TABLE[0]
    assert math.isnan(formats.E8M0_TABLE[255])


def test_e4m3_against_torch_float8():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = formats.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])


def test_e4m3_landmarks_fixture():
    for hx, val in read_golden("e4m3_values.txt"):
        got = formats.E4M3_TABLE[int(hx, 16)]
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_packing_low_nibble_is_even_index():
    codes = np.array([[0x21, 0xF7]], dtype=np.uint8)
    scales = np.array([[127]], dtype=np.uint8)  # 2^0, one block of 32 -> pad
    c = np.zeros((1, 16), dtype=np.uint8)
    c[0, :2] = codes[0]
    w = formats.dequant(c, scales, 1.0, "mxfp4")
    assert list(w[0, :4]) == [0.5, 1.0, 6.0, -6.0]


def _loop_dequant(codes, scales, tscale, fmt):
    rows, half = codes.shape
    K = half * 2
    blk = 32 if fmt == "mxfp4" else 16
    out = np.zeros((rows, K))
    for r in range(rows):
        for i in range(K):
            byte = int(codes[r, i // 2])
            c = byte & 15 if i % 2 == 0 else byte >> 4
            sb = int(scales[r, i // blk])
            if fmt == "mxfp4":
                s = math.ldexp(1.0, sb - 127)
            else:
                e, m = (sb >> 3) & 15, sb & 7
                s = math.ldexp(m / 8, -6) if e == 0 else math.ldexp(1 + m / 8, e - 7)
                s *= float(tscale)
            sign = -1.0 if c & 8 else 1.0
            e2, m2 = (c >> 1) & 3, c & 1
            v = 0.5 * m2 if e2 == 0 else math.ldexp(1 + 0.5 * m2, e2 - 1)
            out[r, i] = sign * v * s
    return out


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_dequant_matches_elementwise_loop(fmt):
    g = np.random.default_rng(3)
    rows, K = 5, 64
    codes = g.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    if fmt == "mxfp4":
        scales = g.integers(110, 140, (rows, K // 32), dtype=np.uint8)
        ts = 1.0
    else:
        scales = g.integers(0, 0x7F, (rows, K // 16), dtype=np.uint8)
        ts = np.float32(2.0 ** -6)
    got = formats.dequant(codes, scales, ts, fmt)
    assert np.array_equal(got, _loop_dequant(codes, scales, ts, fmt))


def test_mxfp8_dequant_against_torch_float8_and_ldexp():
    # E4M3 elements through torch's float8_e4m3fn decoding, times 2^(s - 127)
    g = np.random.default_rng(5)
    rows, K = 6, 96
    codes = g.integers(0, 256, (rows, K), dtype=np.uint8)
    codes[codes & 0x7F == 0x7F] = 0x10   # no NaN codes
    scales = g.integers(100, 150, (rows, K // 32), dtype=np.uint8)
    e = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ref = np.array([[math.ldexp(e[r, i], int(scales[r, i // 32]) - 127) for i in range(K)] for r in range(rows)])
    assert np.array_equal(formats.dequant(codes, scales, 1.0, "mxfp8"), ref)


def test_bf16_dequant_against_torch_bfloat16():
    # little-endian bf16 byte pairs decode as torch's bfloat16 of the same bits
    g = np.random.default_rng(6)
    bits = g.integers(0, 1 << 16, (4, 40), dtype=np.uint16)
    bits[(bits & 0x7F80) == 0x7F80] = 0x3F80   # no inf / NaN
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = formats.dequant(bits.view(np.uint8).reshape(4, 80), np.zeros((4, 0), np.uint8), 1.0, "bf16")
    assert np.array_equal(got, ref)
