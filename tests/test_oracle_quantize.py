"""Pins for the oracle's per-(block, head) absmax FP8 quantiser.

* the absmax element lands exactly on +-448 (code 0x7E / 0xFE);
* an all-zero tile has scale 1 and all-zero codes;
* slots past the valid length are code 0 and do not enter the absmax;
* the reconstruction error obeys the E4M3 half-ulp bound
  |decode(code) * scale - x| <= scale * 2^-4 * |x / scale| (normals) and
  <= scale * 2^-10 (subnormals);
* the scale is the fp32 quotient absmax / 448.
"""
import numpy as np

from oracle import e4m3
from oracle import quantize as QZ


def _tile(seed, bs=16, d=64, outliers=False):
    g = np.random.default_rng(seed)
    x = g.standard_normal((bs, d)).astype(np.float32)
    if outliers:
        m = g.random((bs, d)) < 0.01
        x = np.where(m, x * 20, x).astype(np.float32)
    return x


def test_absmax_element_maps_to_max_code():
    for seed in range(5):
        x = _tile(seed, outliers=True)
        codes, s = QZ.quantize_tile(x, 16)
        i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        assert codes[i] in (0x7E, 0xFE)
        assert s == np.float32(np.max(np.abs(x))) / np.float32(448.0)


def test_zero_tile():
    codes, s = QZ.quantize_tile(np.zeros((16, 64), np.float32), 16)
    assert s == 1.0 and not codes.any()


def test_invalid_slots_are_zero_and_ignored():
    x = _tile(3)
    x[10:] = 1e4          # garbage past the valid length
    codes, s = QZ.quantize_tile(x, 10)
    assert not codes[10:].any()
    assert s == np.float32(np.max(np.abs(x[:10]))) / np.float32(448.0)


def test_reconstruction_error_bound():
    for seed in range(4):
        x = _tile(seed, outliers=True)
        codes, s = QZ.quantize_tile(x, 16)
        y = e4m3.decode(codes) * np.float64(s)
        r = np.abs(x.astype(np.float64) / np.float64(s))
        bound = np.where(r >= 2.0 ** -6, r * 2.0 ** -4, 2.0 ** -10) * np.float64(s)
        # the fp32 division adds at most one fp32 rounding of x / scale
        bound = bound + r * np.float64(s) * 2.0 ** -23
        assert np.all(np.abs(y - x) <= bound)


def test_quantize_blocks_layout():
    g = np.random.default_rng(5)
    cache = g.standard_normal((6, 2, 8, 16)).astype(np.float32)
    codes, scales = QZ.quantize_blocks(cache, [4, 1], [8, 3])
    c41, s41 = QZ.quantize_tile(cache[4, 1], 8)
    assert np.array_equal(codes[4, 1], c41) and scales[4, 1] == s41
    c10, s10 = QZ.quantize_tile(cache[1, 0], 3)
    assert np.array_equal(codes[1, 0], c10) and scales[1, 0] == s10
    assert not codes[0].any() and np.all(scales[0] == 1)


def test_batched_whole_blocks_equal_per_tile_path():
    g = np.random.default_rng(6)
    cache = (g.standard_normal((9, 3, 16, 32)) * np.where(
        g.random((9, 3, 16, 32)) < 0.01, 20, 1)).astype(np.float32)
    cache[4, 1] = 0
    ids = [0, 4, 8, 2]
    codes, scales = QZ.quantize_blocks(cache, ids, [16] * 4)
    for b in ids:
        for h in range(3):
            c, s = QZ.quantize_tile(cache[b, h], 16)
            assert np.array_equal(codes[b, h], c) and scales[b, h] == s
