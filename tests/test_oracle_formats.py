"""Pins of the oracle's number formats against the format definitions and torch.

bf16 widening is checked on all 65,536 bit patterns against torch's own
bfloat16 -> float64 conversion; the E4M3 decoder on all 256 codes against the
OCP specification's code points (golden file) and torch.float8_e4m3fn; the
encoder against torch's round-to-nearest-even conversion on in-range values,
plus saturation, ties, subnormals and decode(encode(x)) = x.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_bf16_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def _golden_e4m3():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_ocp_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            rows.append((int(code, 16), float(val)))
    return rows


def test_e4m3_decode_ocp_code_points():
    for code, val in _golden_e4m3():
        got = oracle.e4m3_to_double(code)
        if math.isnan(val):
            assert math.isnan(got), hex(code)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_e4m3_roundtrip_finite_codes():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        x = oracle.e4m3_to_double(c)
        assert oracle.e4m3_from_float(x) == c, hex(c)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.normal(0, 1, 20000), rng.normal(0, 30, 20000), rng.uniform(-448, 448, 20000),
        rng.uniform(-2**-6, 2**-6, 20000), rng.normal(0, 1e-3, 5000),
        # exact midpoints between neighbouring codes (ties to even)
        [0.5 * (oracle.e4m3_to_double(c) + oracle.e4m3_to_double(c + 1)) for c in range(0, 0x7E)],
    ]).astype(np.float32)
    xs = np.concatenate([xs, -xs])
    xs = xs[np.abs(xs) <= 448]
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_float(float(x)) for x in xs], dtype=np.uint8)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(xs[i]), hex(ref[i]), hex(got[i])) for i in bad[:10]]


def test_e4m3_encode_all_bf16_in_range_match_torch():
    bits = np.arange(65536, dtype=np.uint16)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float()
    keep = torch.isfinite(x) & (x.abs() <= 448)
    x = x[keep]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_float(float(v)) for v in x.numpy()], dtype=np.uint8)
    assert np.array_equal(ref, got)


@pytest.mark.parametrize("x,code", [
    (448.0, 0x7E), (449.0, 0x7E), (464.0, 0x7E), (1e6, 0x7E), (math.inf, 0x7E),
    (-500.0, 0xFE), (-math.inf, 0xFE),
    (2.0**-9, 0x01), (2.0**-10, 0x00), (1.5 * 2.0**-10, 0x01), (-2.0**-11, 0x80),
    (1.0625, 0x38), (1.1875, 0x3A), (0.0, 0x00), (-0.0, 0x80),
])
def test_e4m3_encode_special_cases(x, code):
    # saturation to 448, ties to even, subnormal rounding, signed zero
    assert oracle.e4m3_from_float(x) == code


def test_e4m3_encode_nan():
    assert (oracle.e4m3_from_float(math.nan) & 0x7F) == 0x7F


def test_e4m3_encode_monotone():
    xs = np.linspace(-448, 448, 40001).astype(np.float32)
    vals = [oracle.e4m3_to_double(oracle.e4m3_from_float(float(x))) for x in xs]
    assert all(a <= b for a, b in zip(vals, vals[1:]))


def test_quantize_is_ieee_single_division_then_rne():
    rng = np.random.default_rng(11)
    x = torch.from_numpy(rng.normal(0, 2, 4000).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    for scale in (1.0, 0.0123, 5.5 / 448, 3.0):
        q = (x.float() / torch.tensor(scale, dtype=torch.float32))
        keep = q.abs() <= 448
        ref = q[keep].to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = np.array([oracle.e4m3_quantize(int(b), scale) for b in bits[keep.numpy()]],
                       dtype=np.uint8)
        assert np.array_equal(ref, got), scale
