"""Pins of the oracle's number formats: bf16/fp16 decoding, the int8 code
(round half to even, saturation) and the E4M3 encoder, against library
routines, the format definitions and hand-derived points."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_bf16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([O.bf16_to_f32(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([O.f16_to_f32(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_int8_code_matches_numpy_rint_and_clip():
    rng = np.random.default_rng(0)
    ys = np.concatenate([
        rng.uniform(-300, 300, 20000).astype(np.float32),
        np.arange(-140, 140, dtype=np.float32) + np.float32(0.5),   # exact ties
        np.arange(-140, 140, dtype=np.float32),                     # integers
        np.nextafter(np.arange(-130, 130, dtype=np.float32) + np.float32(0.5), np.float32(0)),
        np.nextafter(np.arange(-130, 130, dtype=np.float32) + np.float32(0.5), np.float32(1e9)),
        np.array([1e30, -1e30, 127.5, -128.5, 127.49999, -128.50002, 0.0, -0.0], np.float32),
    ]).astype(np.float32)
    ref = np.clip(np.rint(ys), -128, 127).astype(np.int8)
    got = np.array([O.int8_code(float(y)) for y in ys], np.int8)
    assert np.array_equal(got, ref)


def test_int8_ties_go_to_even():
    for n in range(-127, 127):
        code = O.int8_code(n + 0.5)
        assert code in (n, n + 1) and code % 2 == 0


def _codes_finite():
    return [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([O.e4m3_decode(int(c)) for c in codes], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_encode_decode_roundtrip():
    for c in _codes_finite():
        assert O.e4m3(O.e4m3_decode(c)) == c


def test_e4m3_midpoints_tie_to_even():
    # between adjacent finite codes of one sign the midpoint must go to the
    # code whose mantissa is even, i.e. the even code
    for sign in (0x00, 0x80):
        for c in range(0, 0x7E):
            lo, hi = O.e4m3_decode(sign | c), O.e4m3_decode(sign | (c + 1))
            mid = np.float32((np.float64(lo) + np.float64(hi)) / 2)
            assert float(mid) == (lo + hi) / 2          # exact in binary32
            want = sign | (c if c % 2 == 0 else c + 1)
            assert O.e4m3(float(mid)) == want, (hex(sign | c), float(mid))


def test_e4m3_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    mag = np.exp2(rng.uniform(-14, math.log2(448), 50000)).astype(np.float32)
    x = (mag * rng.choice([-1, 1], mag.size)).astype(np.float32)
    x = np.concatenate([x, np.linspace(-448, 448, 20001, dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.e4m3(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_golden_points():
    n = 0
    with open(os.path.join(GOLDEN, "e4m3_points.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            val, code = line.split()[:2]
            x = float(val)
            assert O.e4m3(x) == int(code, 16), line
            n += 1
    assert n >= 25
