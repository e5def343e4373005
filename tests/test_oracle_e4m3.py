"""Pins for the oracle's E4M3 codec (CPU only).

The codec is checked against things other than itself: the format's
published code values (tests/golden/e4m3_codes.txt), PyTorch's own
float8_e4m3fn conversion (a library routine) and closed forms of
round-to-nearest-even and saturation.
"""

import os

import numpy as np
import pytest
import torch

from oracle import e4m3
from oracle import paged_attention as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_codes.txt")


def _golden():
    rows = []
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                code, val = line.split()[:2]
                rows.append((int(code, 16), float(val)))
    return rows


def test_golden_codes_decode():
    for code, val in _golden():
        got = e4m3.decode(np.array([code], dtype=np.uint8))[0]
        if np.isnan(val):
            assert np.isnan(got), hex(code)
        else:
            assert got == val and np.signbit(got) == np.signbit(val), hex(code)


def test_golden_codes_encode():
    for code, val in _golden():
        if np.isnan(val):
            assert e4m3.is_nan_code(e4m3.encode(np.array([val])))[0]
        else:
            assert e4m3.encode(np.array([val]))[0] == code, hex(code)


def test_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3.decode(codes)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(lib[~nan]))
    assert nan.sum() == 2


def test_roundtrip_all_finite_codes():
    codes = np.arange(256, dtype=np.uint8)
    finite = ~e4m3.is_nan_code(codes)
    assert np.array_equal(e4m3.encode(e4m3.decode(codes[finite])), codes[finite])


def _all_f16_and_bf16_as_f32():
    bits = np.arange(1 << 16, dtype=np.uint32)
    f16 = bits.astype(np.uint16).view(np.float16).astype(np.float32)
    bf16 = (bits << 16).view(np.float32)
    return np.concatenate([f16, bf16])


def test_encode_matches_torch_in_range():
    # Every fp16 and every bf16 value (all inputs the write path sees), plus
    # random float32.  torch rounds to nearest-even but does not saturate: it
    # gives NaN from 464 up, so compare below that and pin saturation apart.
    x = np.concatenate([_all_f16_and_bf16_as_f32(),
                        np.random.default_rng(0).standard_normal(200000).astype(np.float32) * 50])
    x = x[np.isfinite(x) & (np.abs(x) < 464.0)]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = e4m3.encode(x.astype(np.float64))
    assert np.array_equal(ours, lib)


def test_encode_saturates():
    x = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e6, np.inf, -464.0, -np.inf])
    want = np.array([0x7E] * 7 + [0xFE, 0xFE], dtype=np.uint8)
    assert np.array_equal(e4m3.encode(x), want)


def test_encode_ties_to_even_and_underflow():
    one, step = 1.0, 0.125
    # halfway between 1.0 (0x38, even) and 1.125 (0x39): goes down to 0x38
    assert e4m3.encode(np.array([one + step / 2]))[0] == 0x38
    # halfway between 1.125 (0x39) and 1.25 (0x3A, even): goes up
    assert e4m3.encode(np.array([one + 1.5 * step]))[0] == 0x3A
    # half the smallest subnormal is a tie between 0 and 2^-9: even (zero)
    assert e4m3.encode(np.array([2.0 ** -10]))[0] == 0x00
    assert e4m3.encode(np.array([-(2.0 ** -10)]))[0] == 0x80
    # just above the tie rounds up to the smallest subnormal
    assert e4m3.encode(np.array([2.0 ** -10 * 1.0001]))[0] == 0x01
    assert e4m3.encode(np.array([-0.0]))[0] == 0x80


def test_nan_encodes_to_nan():
    assert e4m3.is_nan_code(e4m3.encode(np.array([np.nan, -np.nan]))).all()


def test_fp8_quantise_is_f32_divide_then_round():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(50000).astype(np.float32)
    bits16 = x.astype(np.float16).view(np.uint16)
    scale = np.float32(4.37 / 448.0)
    got = ref.fp8_quantise(bits16, "f16", scale)
    # library path: torch float32 divide, torch RN-even e4m3 conversion
    t = torch.from_numpy(bits16.view(np.float16)).float() / torch.tensor(scale, dtype=torch.float32)
    lib = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, lib)
    # and the dequantised value is within half an E4M3 step (relative 2^-4) of x / 1
    back = ref.fp8_dequantise(got, scale)
    xs = bits16.view(np.float16).astype(np.float64)
    ok = np.abs(xs) > 2.0 ** -6 * float(scale)
    assert np.all(np.abs(back[ok] - xs[ok]) <= np.abs(xs[ok]) * 2.0 ** -4 * 1.0000001)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_widen_matches_torch(dtype):
    rng = np.random.default_rng(2)
    vals = rng.standard_normal(1000).astype(np.float32) * 10
    td = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    it = {"f16": torch.int16, "bf16": torch.int16, "f32": torch.int32}[dtype]
    t = torch.from_numpy(vals).to(td)
    bits = t.view(it).numpy().view(ref.STORAGE[dtype])
    assert np.array_equal(ref.widen(bits, dtype), t.to(torch.float64).numpy())
