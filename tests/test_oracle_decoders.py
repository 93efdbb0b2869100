"""Pins of the oracle's format decoders and FP16 encoder.

The decoders are written from the bit splits in the "Tensor Core" chapter, table
"精度：FP16、BF16、TF32、FP8" (FP16 1/5/10, BF16 1/8/7, E4M3 1/4/3).  They are
checked exhaustively against independent library decoders (numpy float16, torch
bfloat16 and float8_e4m3fn) and on spot values with closed forms.
"""
import math

import numpy as np
import pytest
import torch


def _same(a, b):
    return (math.isnan(a) and math.isnan(b)) or (a == b and math.copysign(1, a) == math.copysign(1, b))


def test_f16_exhaustive(orc):
    lib_vals = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    for code in range(65536):
        assert _same(orc.decode_f16(code), float(lib_vals[code])), hex(code)


def test_bf16_exhaustive(orc):
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    lib_vals = codes.to(torch.float64).numpy()
    for code in range(65536):
        assert _same(orc.decode_bf16(code), float(lib_vals[code])), hex(code)


def test_e4m3_exhaustive(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    lib_vals = codes.to(torch.float64).numpy()
    for code in range(256):
        assert _same(orc.decode_e4m3(code), float(lib_vals[code])), hex(code)


@pytest.mark.parametrize("code,value", [
    (0x7E, 448.0), (0xFE, -448.0), (0x01, 2.0 ** -9), (0x08, 2.0 ** -6), (0x38, 1.0),
    (0x00, 0.0), (0x77, 240.0), (0x07, 7 * 2.0 ** -9)])
def test_e4m3_spot(orc, code, value):
    assert orc.decode_e4m3(code) == value


def test_e4m3_nan_codes_and_no_inf(orc):
    nans = [c for c in range(256) if math.isnan(orc.decode_e4m3(c))]
    assert nans == [0x7F, 0xFF]
    assert all(math.isfinite(orc.decode_e4m3(c)) for c in range(256) if c not in (0x7F, 0xFF))
    assert math.copysign(1.0, orc.decode_e4m3(0x80)) == -1.0


@pytest.mark.parametrize("code,value", [(0x7BFF, 65504.0), (0x0001, 2.0 ** -24), (0x0400, 2.0 ** -14),
                                        (0x3C00, 1.0), (0xC000, -2.0), (0x7C00, math.inf)])
def test_f16_spot(orc, code, value):
    assert orc.decode_f16(code) == value


def test_f16_encoder_roundtrip(orc):
    for code in range(65536):
        v = orc.decode_f16(code)
        if math.isnan(v):
            continue
        assert orc.encode_f16_rn(v) == code, hex(code)


def test_f16_encoder_ties_to_even(orc):
    # midpoints between neighbouring finite halves go to the even code
    for code in list(range(0, 0x7BFF, 97)) + [0x03FF, 0x0400, 0x3BFF, 0x7BFE]:
        lo, hi = orc.decode_f16(code), orc.decode_f16(code + 1)
        mid = (lo + hi) / 2  # exact in double
        want = code if code % 2 == 0 else code + 1
        assert orc.encode_f16_rn(mid) == want
        assert orc.encode_f16_rn(-mid) == want | 0x8000
    # halfway between the largest finite half and 2^16 overflows to inf
    assert orc.encode_f16_rn(65520.0) == 0x7C00
    assert orc.encode_f16_rn(65519.99) == 0x7BFF


def test_f16_encoder_vs_numpy(orc):
    rng = np.random.default_rng(11)
    vals = np.concatenate([rng.uniform(-70000, 70000, 3000), rng.standard_normal(3000) * 1e-5,
                           rng.standard_normal(3000)]).astype(np.float32)
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).view(np.uint16)
    for v, w in zip(vals, want):
        assert orc.encode_f16_rn(float(v)) == int(w), float(v)


def test_e5m2_exhaustive(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e5m2)
    lib_vals = codes.to(torch.float64).numpy()
    for code in range(256):
        assert _same(orc.decode_e5m2(code), float(lib_vals[code])), hex(code)


@pytest.mark.parametrize("code,value", [(0x7B, 57344.0), (0x01, 2.0 ** -16), (0x04, 2.0 ** -14),
                                        (0x3C, 1.0), (0x7C, math.inf), (0xFC, -math.inf)])
def test_e5m2_spot(orc, code, value):
    assert orc.decode_e5m2(code) == value
