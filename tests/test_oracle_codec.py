"""Pins for the oracle's scalar codecs (fp8 e4m3 / e5m2, int8).

The oracle restates the scalar fp8 quantise / dequantise of the vllm PR 39445
page (Breakdown item 1, Key files: fp8e4m3_to_float_scalar,
float_to_fp8e4m3_scalar) and the int8 round-and-clamp of the vllm PR 38378
page (Breakdown item 3, Review).  Each test pins it to something other than
itself: the OCP FP8 specification's printed values (tests/golden/), torch's
own fp8 casts and rounding, and closed-form properties.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ocp_fp8_values.txt")
FMTS = {"e4m3": (oracle.E4M3, torch.float8_e4m3fn, 0x7E, 448.0),
        "e5m2": (oracle.E5M2, torch.float8_e5m2, 0x7B, 57344.0)}


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                fmt, code, val = line.split()
                rows.append((fmt, int(code, 16), val))
    return rows


def _parse_value(s):
    if s == "nan":
        return math.nan
    if s in ("inf", "-inf"):
        return float(s)
    if s == "-0":
        return -0.0
    sign = -1.0 if s.startswith("-") else 1.0
    s = s.lstrip("-")
    if "*2^" in s:
        m, e = s.split("*2^")
        return sign * float(m) * 2.0 ** int(e)
    if s.startswith("2^"):
        return sign * 2.0 ** int(s[2:])
    return sign * float(s)


@pytest.mark.parametrize("fmt,code,val", _golden_rows())
def test_fp8_decode_spec_values(fmt, code, val):
    got = oracle.fp8_decode(FMTS[fmt][0], code)
    want = _parse_value(val)
    if math.isnan(want):
        assert math.isnan(got)
    else:
        assert got == want and math.copysign(1, got) == math.copysign(1, want)


@pytest.mark.parametrize("fmt", list(FMTS))
def test_fp8_decode_all_codes_match_torch(fmt):
    ofmt, tdt, _, _ = FMTS[fmt]
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(tdt).to(torch.float64).numpy()
    got = np.array([oracle.fp8_decode(ofmt, c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def _finite_codes(fmt):
    max_code = FMTS[fmt][2]
    return list(range(0, max_code + 1)) + list(range(0x80, 0x80 + max_code + 1))


@pytest.mark.parametrize("fmt", list(FMTS))
def test_fp8_encode_round_trip(fmt):
    ofmt = FMTS[fmt][0]
    for c in _finite_codes(fmt):
        assert oracle.fp8_encode(ofmt, oracle.fp8_decode(ofmt, c)) == c, hex(c)


def _torch_cast(fmt, y):
    return (torch.from_numpy(np.asarray(y, np.float32)).to(FMTS[fmt][1])
            .view(torch.uint8).numpy())


@pytest.mark.parametrize("fmt", list(FMTS))
def test_fp8_encode_in_range_matches_torch(fmt):
    ofmt, _, _, vmax = FMTS[fmt]
    rng = np.random.default_rng(7)
    ys = np.concatenate([
        rng.uniform(-vmax, vmax, 3000),
        rng.standard_normal(3000) * rng.choice([1e-4, 1e-2, 1, 10, 100], 3000),
        rng.standard_normal(500) * 2.0 ** -12,
    ]).astype(np.float32)
    ys = ys[np.abs(ys) <= vmax]
    got = oracle.fp8_encode_array(ofmt, ys)
    assert np.array_equal(got, _torch_cast(fmt, ys))


@pytest.mark.parametrize("fmt", list(FMTS))
def test_fp8_encode_midpoints_go_to_even(fmt):
    """Exact midpoints between neighbouring codes round to the even code;
    one float32 ulp to either side rounds to the nearer code."""
    ofmt, tdt, max_code, _ = FMTS[fmt]
    vals = torch.arange(max_code + 1, dtype=torch.int32).to(torch.uint8).view(tdt)
    vals = vals.to(torch.float64).numpy()
    for c in range(max_code):
        mid = np.float32((vals[c] + vals[c + 1]) / 2)
        assert float(mid) == (vals[c] + vals[c + 1]) / 2  # exact in fp32
        even = c if c % 2 == 0 else c + 1
        for sign, sbit in ((1, 0), (-1, 0x80)):
            assert oracle.fp8_encode(ofmt, sign * mid) == even | sbit
            lo = np.nextafter(mid, np.float32(0))
            hi = np.nextafter(mid, np.float32(np.inf))
            assert oracle.fp8_encode(ofmt, sign * lo) == c | sbit
            assert oracle.fp8_encode(ofmt, sign * hi) == (c + 1) | sbit
        assert _torch_cast(fmt, [mid])[0] == even


@pytest.mark.parametrize("fmt", list(FMTS))
def test_fp8_encode_saturates(fmt):
    """Beyond the largest finite value the code saturates (satfinite);
    infinities too.  Largest values: 448 (E4M3), 57344 (E5M2)."""
    ofmt, _, max_code, vmax = FMTS[fmt]
    for y in (vmax, vmax * 1.0001, vmax * 1.07, vmax * 1.2, vmax * 4, 3e38,
              math.inf):
        assert oracle.fp8_encode(ofmt, y) == max_code
        assert oracle.fp8_encode(ofmt, -y) == max_code | 0x80


@pytest.mark.parametrize("fmt", list(FMTS))
def test_fp8_encode_signed_zero(fmt):
    ofmt = FMTS[fmt][0]
    tiny = 2.0 ** -30
    assert oracle.fp8_encode(ofmt, 0.0) == 0x00
    assert oracle.fp8_encode(ofmt, -0.0) == 0x80
    assert oracle.fp8_encode(ofmt, tiny) == 0x00
    assert oracle.fp8_encode(ofmt, -tiny) == 0x80
    assert oracle.fp8_encode(ofmt, 1e-45) == 0x00  # fp32 subnormal


def test_fp8_encode_subnormal_steps():
    """E4M3 subnormals are multiples of 2^-9, E5M2's of 2^-16."""
    for m in range(1, 8):
        assert oracle.fp8_encode(oracle.E4M3, m * 2.0 ** -9) == m
    for m in range(1, 4):
        assert oracle.fp8_encode(oracle.E5M2, m * 2.0 ** -16) == m


def test_int8_ties_and_clamp():
    cases = {0.5: 0, 1.5: 2, 2.5: 2, -0.5: 0, -1.5: -2, -2.5: -2, 0.49: 0,
             0.51: 1, 126.5: 126, 127.4: 127, 127.5: 127, 1000.0: 127,
             -127.5: -128, -128.5: -128, -1e9: -128, 3e38: 127, -0.0: 0}
    for y, want in cases.items():
        assert oracle.int8_encode(y) == want, y


def test_int8_matches_torch_round_half_even():
    rng = np.random.default_rng(3)
    ys = np.concatenate([rng.uniform(-140, 140, 4000),
                         np.arange(-260, 261) / 2.0]).astype(np.float32)
    ref = torch.round(torch.from_numpy(ys)).clamp(-128, 127).to(torch.int8)
    got = np.array([oracle.int8_encode(float(y)) for y in ys], dtype=np.int8)
    assert np.array_equal(got, ref.numpy())


def test_row_bytes():
    assert oracle.row_bytes(oracle.AUTO, 128) == 256
    assert oracle.row_bytes(oracle.FP8_E4M3, 128) == 128
    assert oracle.row_bytes(oracle.FP8_E5M2, 64) == 64
    assert oracle.row_bytes(oracle.INT8_PER_TOKEN_HEAD, 128) == 144
    assert oracle.row_bytes(oracle.FP8_PER_TOKEN_HEAD, 256) == 272
    assert oracle.row_bytes(oracle.FP8_E5M2_PER_TOKEN_HEAD, 128) == 144


def _nearest_code_brute(values: np.ndarray, y: np.ndarray) -> np.ndarray:
    """Nearest of the non-negative finite code values (index = code) to
    |y|, ties to the even code, saturating; sign bit copied.  A plain scan
    over every code in binary64, independent of the oracle's bisection."""
    a = np.abs(y.astype(np.float64))[:, None]
    d = np.abs(values[None, :] - a)
    best = d.min(axis=1, keepdims=True)
    codes = np.arange(values.size)
    cand = np.where(d == best, codes[None, :], 10 ** 6)
    # among equidistant codes (at most two) keep the even one
    even = np.where((cand % 2 == 0) & (cand < 10 ** 6), cand, 10 ** 6).min(axis=1)
    pick = np.where(even < 10 ** 6, even, cand.min(axis=1))
    pick = np.where(a[:, 0] >= values[-1], values.size - 1, pick)
    return (pick | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


@pytest.mark.parametrize("fmt", list(FMTS))
def test_fp8_encode_matches_brute_force_scan(fmt):
    """Every finite bf16 value divided by a handful of scales (the quotients
    the cache writer encodes) against a plain scan of all codes."""
    ofmt, _, _, _ = FMTS[fmt]
    max_code = 0x7E if ofmt == oracle.E4M3 else 0x7B
    values = np.array([oracle.fp8_decode(ofmt, c) for c in range(max_code + 1)])
    bits = np.arange(1 << 16, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    x = x[np.isfinite(x)]
    for s in (1.0, 0.0371, 1.0 / 448.0, 3.3e-5):
        y = (x / np.float32(s)).astype(np.float32)
        y = y[np.isfinite(y)]
        got = oracle.fp8_encode_array(ofmt, y)
        assert np.array_equal(got, _nearest_code_brute(values, y)), s
