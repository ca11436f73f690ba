"""Pins of the oracle's e4m3 codec (CPU only).

The codec is pinned to things other than itself: the OCP E4M3 special values
(golden fixture), torch's float8_e4m3fn (an independent library implementation
of the same format), round-trip and monotonicity invariants, and the format's
half-spacing error bound.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            a, b = line.split()[:2]
            rows.append((a, b))
    return rows


def _torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_special_values(oracle):
    for code_s, val_s in _read_table("e4m3_special_values.txt"):
        code = int(code_s, 16)
        got = oracle.e4m3_to_double(code)
        if val_s == "nan":
            assert math.isnan(got), hex(code)
        else:
            want = float(val_s)
            assert got == want, (hex(code), got, want)
            assert math.copysign(1.0, got) == math.copysign(1.0, want), hex(code)


def test_decode_all_codes_match_torch(oracle):
    ref = _torch_decode_all()
    got = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    assert nan.sum() == 2  # only 0x7f and 0xff


def test_encode_roundtrip_all_codes(oracle):
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_encode_golden_rounding_cases(oracle):
    for x_s, code_s in _read_table("e4m3_rounding_cases.txt"):
        x = np.float32(float(x_s))
        got = oracle.e4m3_from_float(x)
        assert got == int(code_s, 16), (x_s, hex(got), code_s)


def test_encode_matches_torch_below_overflow(oracle):
    """torch rounds to nearest-even but sends |x| >= 464 to NaN; compare below."""
    rng = np.random.Generator(np.random.PCG64(1))
    bits = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 464.0)]
    # add every midpoint and its fp32 neighbours, where ties are decided
    mags = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    extra = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                            np.nextafter(mids, np.float32(1e9)), mags.astype(np.float32)])
    extra = np.concatenate([extra, -extra]).astype(np.float32)
    x = np.concatenate([x, extra])
    # also dense normal samples at the scales the cache sees
    x = np.concatenate([x, (rng.standard_normal(200_000) * 100).astype(np.float32)])
    x = x[np.abs(x) < 464.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(ref[i])) for i in bad[:10]]


def test_encode_saturates_and_nan(oracle):
    for v in [448.0, 448.5, 463.9, 464.0, 500.0, 3.4e38, float("inf")]:
        assert oracle.e4m3_from_float(v) == 0x7E
        assert oracle.e4m3_from_float(-v) == 0xFE
    assert oracle.e4m3_from_float(float("nan")) == 0x7F


def test_encode_monotone_and_error_bound(oracle):
    x = np.linspace(-448.0, 448.0, 2_000_001, dtype=np.float64).astype(np.float32)
    codes = oracle.e4m3_encode(x)
    y = oracle.e4m3_decode(codes)
    assert np.all(np.diff(y) >= 0)
    # half the local spacing: 2^(e-7-3)/2 for normals, 2^-10 for subnormals
    ax = np.abs(x.astype(np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -6)))
    half = np.where(ax < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 3) / 2)
    assert np.all(np.abs(y - x) <= half * (1 + 1e-12))
