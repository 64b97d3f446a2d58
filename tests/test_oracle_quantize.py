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


# ---------------------------------------------------------------- append ---
def _fill(x, order):
    """Append the rows of x (fp32 [bs, d]) in the given order of offsets...
    offsets stay 0, 1, 2, ... (the block fills in order); ``order`` permutes
    which row of x arrives at each offset.  Returns (codes, scale, rows)."""
    bs, d = x.shape
    codes = np.full((bs, d), 0x55, dtype=np.uint8)   # stale bytes of a reused block
    scale = np.float32(123.0)                        # stale scale
    rows = x[order]
    for off in range(bs):
        codes, scale = QZ.append_token(codes, scale, off, rows[off])
    return codes, scale, rows


def test_append_in_falling_absmax_order_equals_whole_block_quantiser():
    for seed in range(4):
        x = _tile(seed, outliers=True)
        order = np.argsort(-np.max(np.abs(x), axis=1), kind="stable")
        codes, scale, rows = _fill(x, order)
        c_ref, s_ref = QZ.quantize_tile(rows, len(rows))
        assert scale == s_ref and np.array_equal(codes, c_ref)


def test_append_final_scale_is_whole_block_scale_in_any_order():
    for seed in range(4):
        x = _tile(seed, outliers=True)
        order = np.random.default_rng(seed).permutation(len(x))
        _, scale, rows = _fill(x, order)
        assert scale == QZ.block_scale(rows)


def test_append_first_token_resets_a_stale_block():
    x = _tile(7)[0]
    codes, s = QZ.append_token(np.full((16, 64), 0x7E, np.uint8), np.float32(1e-9), 0, x)
    c_ref, s_ref = QZ.quantize_tile(x[None, :], 1)
    assert s == s_ref and np.array_equal(codes[0], c_ref[0])
    assert np.array_equal(codes[1:], np.full((15, 64), 0x7E, np.uint8))  # untouched
    z, s0 = QZ.append_token(codes, s, 0, np.zeros(64, np.float32))
    assert s0 == 1.0 and not z[0].any()


def test_append_without_growth_keeps_earlier_codes():
    x = _tile(8)
    codes, s = QZ.quantize_tile(x, 10)
    small = x[3] * np.float32(0.5)                   # absmax below the block's
    c2, s2 = QZ.append_token(codes, s, 10, small)
    assert s2 == s and np.array_equal(c2[:10], codes[:10])
    assert np.array_equal(c2[10], e4m3.encode_fast((small / s).astype(np.float32)))


def test_append_growth_requantises_within_two_roundings():
    x = _tile(9)
    codes, s = QZ.quantize_tile(x, 12)
    big = x[0] * np.float32(9.0)                     # new absmax: the scale grows
    c2, s2 = QZ.append_token(codes, s, 12, big)
    assert s2 == np.float32(np.max(np.abs(big)) / np.float32(448.0)) and s2 > s
    i = np.argmax(np.abs(big))
    assert c2[12, i] in (0x7E, 0xFE)                 # the new absmax lands on 448
    y = e4m3.decode(c2[:12]) * np.float64(s2)
    r = np.abs(x[:12].astype(np.float64))
    # first rounding at the old scale, second at the new (each half an ulp
    # of a 3-bit mantissa, or the subnormal step)
    b1 = np.maximum(r * 2.0 ** -4, np.float64(s) * 2.0 ** -10)
    b2 = np.maximum((r + b1) * 2.0 ** -4, np.float64(s2) * 2.0 ** -10)
    assert np.all(np.abs(y - r * np.sign(x[:12])) <= b1 + b2 + r * 2.0 ** -20)
    assert np.array_equal(c2[13:], codes[13:])


def test_cache_write_fp8_layout_and_skip():
    g = np.random.default_rng(12)
    nb, hkv, bs, d = 5, 2, 8, 16
    kc = np.zeros((nb, hkv, bs, d), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.ones((nb, hkv), np.float32)
    vs = np.ones_like(ks)
    kn = g.standard_normal((3, hkv, d)).astype(np.float32)
    vn = g.standard_normal((3, hkv, d)).astype(np.float32)
    slots = np.array([3 * bs + 0, -1, 3 * bs + 1])
    k2, v2, ks2, vs2 = QZ.cache_write_fp8(kn, vn, slots, kc, vc, ks, vs)
    for h in range(hkv):
        c, s = QZ.append_token(kc[3, h], ks[3, h], 0, kn[0, h])
        c, s = QZ.append_token(c, s, 1, kn[2, h])
        assert np.array_equal(k2[3, h], c) and ks2[3, h] == s
    assert not k2[[0, 1, 2, 4]].any() and np.all(ks2[[0, 1, 2, 4]] == 1)
