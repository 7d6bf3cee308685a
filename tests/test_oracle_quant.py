"""Pins of the oracle's activation quantisers (no GPU): round trips, the
spec's tie rule, an independent threshold encoder and torch's float8 rounding."""
import math

import numpy as np
import pytest
import torch

from conftest import ORACLES, read_golden, swap_oracle
from oracle import formats, quant


@pytest.fixture(autouse=True, params=ORACLES)
def oracle_impl(request, monkeypatch):
    return swap_oracle(__name__, request, monkeypatch, ("formats", "quant"))



def test_e2m1_roundtrip_all_codes():
    for c in range(16):
        assert quant.e2m1_encode(np.array([formats.E2M1_TABLE[c]]))[0] == c


def test_e2m1_rounding_fixture():
    for v, c in read_golden("e2m1_rounding.txt"):
        assert quant.e2m1_encode(np.array([float(v)]))[0] == int(c), v


def _threshold_encode(v):
    # independent formulation: compare against the midpoints, the even side
    # of each midpoint is inclusive (0, 1.0, 2.0, 4.0 have mantissa bit 0)
    a = abs(v)
    if a <= 0.25:
        c = 0
    elif a < 0.75:
        c = 1
    elif a <= 1.25:
        c = 2
    elif a < 1.75:
        c = 3
    elif a <= 2.5:
        c = 4
    elif a < 3.5:
        c = 5
    elif a <= 5.0:
        c = 6
    else:
        c = 7
    return c | (8 if math.copysign(1.0, v) < 0 else 0)


def test_e2m1_encode_vs_threshold_encoder():
    g = np.random.default_rng(5)
    v = np.concatenate([g.standard_normal(4000) * 3, g.uniform(-8, 8, 4000),
                        np.arange(-7, 7.01, 0.125)])
    got = quant.e2m1_encode(v)
    assert [int(x) for x in got] == [_threshold_encode(float(x)) for x in v]


def test_e4m3_encode_vs_torch():
    g = np.random.default_rng(6)
    v = np.concatenate([g.uniform(0, 448, 3000), np.exp(g.uniform(-12, 6, 3000)),
                        formats.E4M3_TABLE[:0x7F]])
    v = v[v <= 448].astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = quant.e4m3_encode_satfinite(v.astype(np.float64))
    assert np.array_equal(got, ref)
    assert quant.e4m3_encode_satfinite(np.array([500.0, 1e9]))[0] == 0x7E


def test_mxfp4_scale_exponent_is_floor_log2_minus_2():
    g = np.random.default_rng(7)
    v = (g.standard_normal((16, 64)) * np.exp(g.uniform(-20, 20, (16, 1)))).astype(np.float32)
    _, s = quant.quant_mxfp4(v)
    for r in range(16):
        for b in range(2):
            amax = float(np.abs(v[r, 32 * b:32 * b + 32]).max())
            m, ex = math.frexp(amax)
            assert int(s[r, b]) - 127 == (ex - 1) - 2


def test_mxfp4_exact_roundtrip_of_grid_values():
    # blocks of E2M1 grid values times 2^X whose largest magnitude is 4 or 6
    # quantise back to exactly the same codes and exponent
    g = np.random.default_rng(8)
    rows, K = 6, 96
    codes = g.integers(0, 16, (rows, K)).astype(np.uint8)
    codes[:, ::32] = np.where(g.integers(0, 2, (rows, K // 32)) > 0, 7, 6)
    X = g.integers(-30, 30, (rows, K // 32))
    vals = formats.E2M1_TABLE[codes] * np.ldexp(1.0, np.repeat(X, 32, axis=1))
    packed, s = quant.quant_mxfp4(vals)
    assert np.array_equal(s.astype(int) - 127, X)
    assert np.array_equal(formats.unpack_codes(packed), codes)


def test_mxfp4_zero_block():
    packed, s = quant.quant_mxfp4(np.zeros((1, 32)))
    assert s[0, 0] == 0 and not packed.any()


def test_nvfp4_exact_roundtrip_of_grid_values():
    g = np.random.default_rng(9)
    rows, K = 4, 64
    codes = g.integers(0, 16, (rows, K)).astype(np.uint8)
    codes[:, ::16] = 7                                 # |6| sets the block amax
    sb = g.integers(0x08, 0x70, (rows, K // 16)).astype(np.uint8)  # normal E4M3
    gs = 0.5
    vals = formats.E2M1_TABLE[codes] * np.repeat(formats.E4M3_TABLE[sb], 16, axis=1) * gs
    packed, s = quant.quant_nvfp4(vals, gs)
    assert np.array_equal(s, sb)
    assert np.array_equal(formats.unpack_codes(packed), codes)


def test_nvfp4_zero_block_and_saturation():
    v = np.zeros((1, 32))
    v[0, 16:] = 1e6
    packed, s = quant.quant_nvfp4(v, 1.0)
    assert s[0, 0] == 0 and s[0, 1] == 0x7E
    c = formats.unpack_codes(packed)
    assert not c[0, :16].any() and (c[0, 16:] == 7).all()


def test_quant_error_bounded_by_half_step():
    # the dequantised value is the nearest grid point: |err| <= half the
    # local E2M1 spacing times the block scale (spacing <= 2 below 6)
    g = np.random.default_rng(10)
    v = g.standard_normal((8, 64))
    packed, s = quant.quant_mxfp4(v)
    w = formats.dequant(packed, s, 1.0, "mxfp4")
    scale = np.repeat(formats.E8M0_TABLE[s], 32, axis=1)
    q = v / scale
    err = np.abs(w - v) / scale
    inside = np.abs(q) <= 6
    assert (err[inside] <= np.where(np.abs(q[inside]) < 2, 0.25, np.where(np.abs(q[inside]) < 4, 0.5, 1.0)) + 1e-12).all()


def test_mxfp8_scale_exponent_and_codes_against_torch():
    # X = floor(log2 amax) - 8 (math.frexp); elements v / 2^X rounded by torch's
    # float8_e4m3fn conversion (nearest even) after clamping to +-448
    g = np.random.default_rng(8)
    v = (g.standard_normal((7, 64)) * np.exp2(g.integers(-20, 20, (7, 1)))).astype(np.float32)
    v[3, :32] = 0.0
    codes, scales = quant.quant_mxfp8(v)
    for r in range(7):
        for b in range(2):
            blk = v[r, 32 * b:32 * (b + 1)].astype(np.float64)
            amax = np.abs(blk).max()
            X = -127 if amax == 0 else math.frexp(amax)[1] - 1 - 8
            assert scales[r, b] == X + 127
            q = np.clip(blk * 2.0 ** -X, -448.0, 448.0).astype(np.float32)
            ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            got = codes[r, 32 * b:32 * (b + 1)]
            nz = q != 0   # torch's sign of a zero result follows the input; compare magnitudes there
            assert np.array_equal(got[nz], ref[nz]) and np.array_equal(got[~nz] & 0x7F, ref[~nz] & 0x7F)


def test_mxfp8_exact_roundtrip_of_grid_values():
    # values on the E4M3 grid times 2^X come back unchanged
    g = np.random.default_rng(9)
    e4 = formats.E4M3_TABLE[:0x7F]
    mags = e4[(e4 >= 2.0 ** -6) & (e4 <= 448)]
    v = g.choice(mags, size=(4, 64)) * g.choice([-1.0, 1.0], size=(4, 64))
    v[:, ::32] = 448.0   # pins the block exponent: floor(log2 448) - 8 = 0
    c, s = quant.quant_mxfp8((v * 2.0 ** -5).astype(np.float32))
    assert np.array_equal(formats.dequant(c, s, 1.0, "mxfp8"), v * 2.0 ** -5)


def test_bf16_rounding_against_torch():
    g = np.random.default_rng(10)
    v = g.standard_normal(2000) * np.exp2(g.integers(-30, 30, 2000))
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(quant.round_bf16(v), ref)
