"""Pins of the oracle's number-format helpers against library conversions and
closed forms (CPU only).

bf16 widening and bf16 round-to-nearest-even are checked against torch's
float32<->bfloat16 casts; e4m3 decoding against torch's float8_e4m3fn cast,
code by code, plus values fixed by the OCP FP8 format definition.
"""
import math
import struct

import numpy as np
import pytest
import torch

import oracle


def _f32_from_bits(b):
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def test_bf16_widen_all_patterns():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float32).numpy()
    for b in range(0, 1 << 16, 7):  # every 7th pattern: all exponents, signs and NaNs
        got = oracle.bf16_to_f32(b)
        r = float(ref[b])
        if math.isnan(r):
            assert math.isnan(got)
        else:
            assert struct.pack("<f", got) == struct.pack("<f", r), hex(b)


@pytest.mark.parametrize("x,expected", [
    (1.0, 0x3F80),
    (1.0 + 2 ** -8, 0x3F80),            # exact midpoint, 1.0 is even
    (1.0 + 3 * 2 ** -8, 0x3F82),        # midpoint between 0x3F81 (odd) and 0x3F82 (even)
    (1.0 + 2 ** -8 + 2 ** -20, 0x3F81),  # just above the midpoint
    (-1.5, 0xBFC0),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (float("inf"), 0x7F80),
    (float("-inf"), 0xFF80),
    (2.0 ** -133, 0x0001),              # smallest bf16 subnormal
    (3.0 * 2 ** -134, 0x0002),          # 1.5 ulps of subnormal: midpoint, rounds to even 2
])
def test_bf16_rne_closed_forms(x, expected):
    assert oracle.f32_to_bf16(x) == expected


def test_bf16_rne_largest_finite_overflows_to_inf():
    # 0x7F7FFFFF is above the midpoint between bf16 max (0x7F7F) and 2^128.
    assert oracle.f32_bits_to_bf16(0x7F7FFFFF) == 0x7F80
    assert oracle.f32_bits_to_bf16(0x7F7F7FFF) == 0x7F7F  # below the midpoint
    assert oracle.f32_bits_to_bf16(0x7F7F8000) == 0x7F80  # midpoint, 0x7F7F is odd


def test_bf16_rne_nan_stays_nan():
    for b in (0x7FC00000, 0x7F800001, 0xFFC12345, 0x7FFFFFFF):
        r = oracle.f32_bits_to_bf16(b)
        assert (r & 0x7F80) == 0x7F80 and (r & 0x7F) != 0
        assert (r >> 15) == (b >> 31)


def test_bf16_rne_matches_torch_on_random_and_tie_patterns():
    rng = np.random.default_rng(1)
    pats = rng.integers(0, 1 << 32, size=6000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 1 << 16, size=2000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    near = (rng.integers(0, 1 << 16, size=2000, dtype=np.uint64).astype(np.uint32) << 16) | \
        rng.choice(np.array([0x7FFF, 0x8001, 0x0001, 0xFFFF], np.uint32), size=2000)
    allp = np.concatenate([pats, ties, near])
    f = allp.view(np.float32)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for i in range(len(allp)):
        if np.isnan(f[i]):
            continue
        assert oracle.f32_bits_to_bf16(int(allp[i])) == int(ref[i]), hex(int(allp[i]))


def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    for c in range(256):
        got = oracle.e4m3_to_f32(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), hex(c)
        else:
            assert got == float(ref[c]) and math.copysign(1, got) == math.copysign(1, ref[c]), hex(c)


@pytest.mark.parametrize("code,value", [
    (0x7E, 448.0),            # S.1111.110: largest finite
    (0x38, 1.0),              # exponent 7 = bias
    (0x01, 2.0 ** -9),        # smallest subnormal
    (0x07, 7 * 2.0 ** -9),    # largest subnormal
    (0x08, 2.0 ** -6),        # smallest normal
    (0xC0, -2.0),
    (0x00, 0.0),
])
def test_e4m3_closed_forms(code, value):
    assert oracle.e4m3_to_f32(code) == value


def test_e4m3_nan_codes():
    assert math.isnan(oracle.e4m3_to_f32(0x7F))
    assert math.isnan(oracle.e4m3_to_f32(0xFF))


def test_f16_widen_all_patterns():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.float16).to(torch.float32).numpy()
    for b in range(1 << 16):
        got = oracle.f16_to_f32(b)
        r = float(ref[b])
        if math.isnan(r):
            assert math.isnan(got), hex(b)
        else:
            assert struct.pack("<f", got) == struct.pack("<f", r), hex(b)


@pytest.mark.parametrize("x,expected", [
    (1.0, 0x3C00), (-2.0, 0xC000), (65504.0, 0x7BFF),
    (65519.0, 0x7BFF),                  # below the midpoint to 65536: stays at the largest finite
    (65520.0, 0x7C00),                  # the midpoint rounds to even, i.e. to infinity
    (2.0 ** -24, 0x0001),               # smallest subnormal
    (2.0 ** -25, 0x0000),               # exactly half of it: ties to even (zero)
    (3 * 2.0 ** -26, 0x0001),           # above half
    (2.0 ** -14, 0x0400),               # smallest normal
    (1.0 + 2.0 ** -11, 0x3C00),         # midpoint, 1.0 is even
    (1.0 + 3 * 2.0 ** -11, 0x3C02),     # midpoint between 0x3C01 and 0x3C02 (even)
    (0.0, 0x0000), (-0.0, 0x8000), (float("inf"), 0x7C00), (float("-inf"), 0xFC00),
])
def test_f16_rne_closed_forms(x, expected):
    assert oracle.f32_bits_to_f16(int(np.array([x], np.float32).view(np.uint32)[0])) == expected


def test_f16_rne_matches_torch_on_random_tie_and_subnormal_patterns():
    rng = np.random.default_rng(2)
    pats = rng.integers(0, 1 << 32, size=4000, dtype=np.uint64).astype(np.uint32)
    # exponents around the binary16 range, including its subnormals and overflow
    exps = rng.integers(127 - 27, 127 + 17, size=6000, dtype=np.uint64).astype(np.uint32)
    mans = rng.integers(0, 1 << 23, size=6000, dtype=np.uint64).astype(np.uint32)
    sgn = rng.integers(0, 2, size=6000, dtype=np.uint64).astype(np.uint32) << 31
    near = sgn | (exps << 23) | mans
    ties = sgn[:3000] | (exps[:3000] << 23) | (mans[:3000] & ~np.uint32(0x1FFF)) | np.uint32(0x1000)
    allp = np.concatenate([pats, near, ties])
    f = allp.view(np.float32)
    ref = torch.from_numpy(f.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    for i in range(len(allp)):
        if np.isnan(f[i]):  # a NaN stays a NaN (exponent all ones, mantissa non-zero)
            r = oracle.f32_bits_to_f16(int(allp[i]))
            assert (r & 0x7C00) == 0x7C00 and (r & 0x3FF) != 0, hex(int(allp[i]))
            continue
        assert oracle.f32_bits_to_f16(int(allp[i])) == int(ref[i]), hex(int(allp[i]))


def test_f16_nan_stays_nan_with_its_sign():
    for b in (0x7FC00000, 0x7F800001, 0xFFC12345, 0x7FFFFFFF, 0xFF800001):
        r = oracle.f32_bits_to_f16(b)
        assert (r & 0x7C00) == 0x7C00 and (r & 0x3FF) != 0, hex(b)
        assert (r >> 15) == (b >> 31)
