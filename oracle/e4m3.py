"""OCP OFP8 E4M3 codec (oracle; test infrastructure only).

Written from the format definition in the OCP "8-bit Floating Point
Specification (OFP8)", E4M3 encoding:

* 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
* exponent field 0 encodes subnormals  (-1)^s * 2^-6 * (m / 8);
* exponent field 1..15 encodes normals (-1)^s * 2^(e-7) * (1 + m / 8);
* S.1111.111 (0x7F / 0xFF) is NaN; there are no infinities, so the largest
  finite magnitude is 2^8 * 1.75 = 448 (code 0x7E).

The encoder rounds to nearest, ties to even, and saturates finite values and
infinities to +-448 ("satfinite" conversion).  NaN encodes as 0x7F.

FP8 caches are the route the page "Paged Attention and KV Cache
Fragmentation" (section "Quantization as a way to stretch paged memory
further") describes for halving the per-token KV footprint.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def decode_code(code: int) -> float:
    """Value of one E4M3 byte, straight from the field definitions."""
    code = int(code) & 0xFF
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        mag = 2.0 ** -6 * (m / 8.0)
    else:
        mag = 2.0 ** (e - 7) * (1.0 + m / 8.0)
    return -mag if s else mag


# 256-entry table, built by calling the scalar definition above.
DECODE_TABLE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)


def decode(codes: np.ndarray) -> np.ndarray:
    """Decode an array of E4M3 bytes (uint8) to float64 values."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def _encode_scalar(x: float) -> int:
    """fp32/fp64 value -> E4M3 byte, RNE, saturating to +-448."""
    if np.isnan(x):
        return NAN_CODE
    sign = 0x80 if np.signbit(x) else 0x00
    a = abs(float(x))
    if a >= E4M3_MAX:          # includes +-inf: satfinite clamps to max finite
        return sign | 0x7E
    if a == 0.0:
        return sign
    # Grid spacing: 2^(e-3) inside binade [2^e, 2^(e+1)), e >= -6; the
    # subnormal range [0, 2^-6) shares the spacing of the first binade, 2^-9.
    e = max(int(np.floor(np.log2(a))), -6)
    # Guard against log2 rounding at exact powers of two.
    if a < 2.0 ** e and e > -6:
        e -= 1
    if a >= 2.0 ** (e + 1):
        e += 1
    ulp = 2.0 ** (e - 3)
    q = np.rint(a / ulp)       # exact division by a power of two; rint is RNE
    v = q * ulp
    if v >= E4M3_MAX:          # rounding up past the largest code saturates
        return sign | 0x7E
    if v < 2.0 ** -6:          # subnormal: v = m * 2^-9, m in 0..7
        m = int(round(v / 2.0 ** -9))
        return sign | m
    ev = int(np.floor(np.log2(v)))
    if v < 2.0 ** ev:
        ev -= 1
    if v >= 2.0 ** (ev + 1):
        ev += 1
    m = int(round(v / 2.0 ** (ev - 3))) - 8
    assert 0 <= m <= 7, (x, v, ev, m)
    return sign | ((ev + 7) << 3) | m


def encode(x: np.ndarray) -> np.ndarray:
    """Encode float values (float32 or exactly-representable float64) to E4M3.

    Element by element through :func:`_encode_scalar`; slow but obviously
    correct.  Use :func:`encode_fast` for large arrays.
    """
    flat = np.asarray(x, dtype=np.float64).ravel()
    out = np.fromiter((_encode_scalar(v) for v in flat), dtype=np.uint8,
                      count=flat.size)
    return out.reshape(np.shape(x))


def encode_fast(x: np.ndarray) -> np.ndarray:
    """Same mapping as :func:`encode`, by nearest-code search over the table.

    For each input the two neighbouring finite codes of the sorted positive
    grid are found with ``searchsorted``; the nearer one wins and exact ties go
    to the code with an even mantissa (even code, since the mantissa is the low
    3 bits).  Magnitudes at or above 448 (and infinities) saturate to 448; NaN
    maps to 0x7F.  Tests check it equals :func:`encode` on every midpoint and
    on random inputs.
    """
    xv = np.asarray(x, dtype=np.float64)
    flat = xv.ravel()
    out = np.empty(flat.size, dtype=np.uint8)
    nan = np.isnan(flat)
    sign = np.where(np.signbit(flat), 0x80, 0x00).astype(np.uint8)
    a = np.abs(np.where(nan, 0.0, flat))
    grid = DECODE_TABLE[:0x7F]                # codes 0x00..0x7E, ascending
    hi = np.searchsorted(grid, a, side="left")  # first grid value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    dlo = a - grid[lo]
    dhi = grid[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    code = np.where(a == grid[hi], hi, code)  # exact hits (incl. 0)
    out[:] = (code.astype(np.uint8) | sign)
    out[nan] = NAN_CODE
    return out.reshape(xv.shape)
