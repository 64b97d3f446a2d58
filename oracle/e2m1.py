"""FP4 E2M1 element codec (oracle; test infrastructure only).

The page "Paged Attention and KV Cache Fragmentation", section "Quantization
as a way to stretch paged memory further", names NVFP4 as the Blackwell KV
format that halves FP8 once more, without defining it.  The element type is
the 4-bit E2M1 float of the OCP Microscaling (MX) specification v1.0 (section
"FP4", the element format NVIDIA's NVFP4 also uses):

    bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa;
    exponent 0 is subnormal: value = mantissa * 0.5;
    otherwise value = 2^(exponent - 1) * (1 + mantissa / 2);
    no infinities and no NaN; the largest magnitude is 6.

Encoding (fp32 -> E2M1) is round to nearest, ties to the even code (mantissa
bit 0), saturating to +-6.  Readings taken where the format leaves the
conversion open, matching what the CUDA conversion API documents:
magnitudes above 6 (and infinities) give +-6; NaN gives +6; the sign is kept
when a value rounds to zero, so a small negative input encodes as -0 (0x8).
"""
from __future__ import annotations

import numpy as np

E2M1_MAX = 6.0


def _decode_code(c: int) -> float:
    s = -1.0 if c & 0x8 else 1.0
    e = (c >> 1) & 0x3
    m = c & 0x1
    if e == 0:
        return s * m * 0.5
    return s * 2.0 ** (e - 1) * (1.0 + m / 2.0)


#: value of each 4-bit code 0x0..0xF (fp64)
DECODE_TABLE = np.array([_decode_code(c) for c in range(16)], dtype=np.float64)


def decode(codes) -> np.ndarray:
    """fp64 value of each 4-bit code (only the low 4 bits are looked at)."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def encode(y) -> np.ndarray:
    """Round each value to the nearest E2M1 code (ties to the even code).

    For each magnitude the two neighbouring codes of the positive grid
    0x0..0x7 are found; the nearer wins and an exact tie goes to the code
    with mantissa bit 0.  Returns uint8 codes 0x0..0xF.
    """
    yv = np.asarray(y, dtype=np.float64)
    flat = yv.ravel()
    nan = np.isnan(flat)
    sign = np.where(np.signbit(flat) & ~nan, 0x8, 0x0).astype(np.uint8)
    a = np.abs(np.where(nan, E2M1_MAX, flat))
    grid = DECODE_TABLE[:8]                       # 0, .5, 1, 1.5, 2, 3, 4, 6
    hi = np.minimum(np.searchsorted(grid, a, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    dlo = a - grid[lo]
    dhi = grid[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= E2M1_MAX, 7, code)
    code = np.where(a == grid[hi], hi, code)
    return (code.astype(np.uint8) | sign).reshape(yv.shape)
