"""Pins for the oracle's E4M3 codec.

* spec values: the OCP OFP8 table (tests/golden/e4m3_spec_values.txt);
* library cross-check: torch's CPU float8_e4m3fn conversion (RNE; NaN above
  the range, so compared only inside +-448) and its decode of all 256 codes;
* round trip, ties-to-even at every midpoint, saturation, NaN;
* the fast table-search encoder equals the scalar one.
"""
import os

import numpy as np
import pytest
import torch

from oracle import e4m3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_spec_values.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        c, v = line.split()
        rows.append((int(c, 16), float(v)))
    return rows


def test_spec_table_values():
    for code, val in _golden():
        got = e4m3.decode_code(code)
        if np.isnan(val):
            assert np.isnan(got), hex(code)
        else:
            assert got == val and np.signbit(got) == np.signbit(val), hex(code)


def test_decode_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3.DECODE_TABLE
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], ours[m])
    assert np.array_equal(np.signbit(ref[m]), np.signbit(ours[m]))


def test_exactly_two_nan_codes_and_max():
    nan_codes = [c for c in range(256) if np.isnan(e4m3.DECODE_TABLE[c])]
    assert nan_codes == [0x7F, 0xFF]
    assert np.nanmax(e4m3.DECODE_TABLE) == 448.0
    assert np.nanmin(e4m3.DECODE_TABLE) == -448.0


def test_round_trip_all_finite_codes():
    for c in range(256):
        v = e4m3.DECODE_TABLE[c]
        if np.isnan(v):
            continue
        assert e4m3._encode_scalar(v) == c, hex(c)


def _positive_midpoints():
    grid = e4m3.DECODE_TABLE[:0x7F]
    return (grid[:-1] + grid[1:]) / 2.0, np.arange(0x7E)


def test_ties_to_even_at_every_midpoint():
    mids, lo = _positive_midpoints()
    for mid, c in zip(mids, lo):
        expect = c if c % 2 == 0 else c + 1
        assert e4m3._encode_scalar(mid) == expect, (mid, c)
        assert e4m3._encode_scalar(-mid) == (expect | 0x80)
        # just off the midpoint rounds to the nearer code
        assert e4m3._encode_scalar(np.nextafter(mid, 0)) == c
        assert e4m3._encode_scalar(np.nextafter(mid, np.inf)) == c + 1


def test_saturation_and_nan():
    for x in (448.0, 449.0, 463.9, 464.0, 500.0, 1e6, np.inf):
        assert e4m3._encode_scalar(x) == 0x7E
        assert e4m3._encode_scalar(-x) == 0xFE
    assert e4m3._encode_scalar(np.nan) == 0x7F
    assert e4m3._encode_scalar(0.0) == 0x00
    assert e4m3._encode_scalar(-0.0) == 0x80
    # below half the smallest subnormal: rounds to (signed) zero
    assert e4m3._encode_scalar(2.0 ** -11) == 0x00
    assert e4m3._encode_scalar(-(2.0 ** -11)) == 0x80


def test_encoder_matches_torch_inside_range():
    g = np.random.default_rng(7)
    x = np.concatenate([
        g.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)
    ]).astype(np.float32)
    mids, _ = _positive_midpoints()
    x = np.concatenate([x, mids.astype(np.float32), -mids.astype(np.float32)])
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = e4m3.encode(x)
    bad = np.nonzero(ref != ours)[0]
    assert bad.size == 0, [(float(x[i]), hex(ref[i]), hex(ours[i])) for i in bad[:5]]


def test_fast_encoder_equals_scalar_encoder():
    g = np.random.default_rng(11)
    x = np.concatenate([
        g.standard_normal(5000) * 100, g.standard_normal(5000) * 1e-3,
        np.array([0.0, -0.0, 448.0, 449.0, 1e9, -1e9, np.inf, -np.inf, np.nan]),
    ]).astype(np.float32)
    mids, _ = _positive_midpoints()
    x = np.concatenate([x, mids.astype(np.float32), -mids.astype(np.float32)])
    assert np.array_equal(e4m3.encode(x), e4m3.encode_fast(x))


@pytest.mark.parametrize("c", [0x01, 0x08, 0x38, 0x7D])
def test_monotone_neighbourhood(c):
    v = e4m3.DECODE_TABLE[c]
    assert e4m3._encode_scalar(np.nextafter(v, np.inf)) == c
    assert e4m3._encode_scalar(np.nextafter(v, 0)) == c
