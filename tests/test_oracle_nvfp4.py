"""Pins for the oracle's FP4 E2M1 codec and NVFP4 cache quantiser.

What fixes each value, independently of the oracle's own code:

* the E2M1 value set is the one printed by the OCP Microscaling Formats
  specification v1.0 (FP4 E2M1: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their
  negatives; largest magnitude 6, no infinity or NaN);
* round-to-nearest-even: each midpoint of that grid goes to the neighbour
  with mantissa bit 0, worked out by hand below; random inputs go to a
  nearest grid value found by brute force over the printed set;
* a hand-worked group (0.75 * i, i = 0..15, S = 1): a = 11.25, block scale
  11.25 / 6 = 1.875 = E4M3 0x3F, y = 0.4 * i, codes by hand;
* lossless round trip: values built as code * 2^k * S with a full-scale
  element in every group quantise back to exactly those codes, so the NVFP4
  decode oracle equals the (separately pinned) dense attention oracle on
  those values;
* the byte layout, by a hand-packed example;
* the NVFP4 footprint the page "Paged Attention and KV Cache Fragmentation"
  prints for Llama 3.1 70B at 128K tokens (about 10.7 GB, a quarter of BF16).
"""
import numpy as np
import pytest

from oracle import e2m1, e4m3, footprint
from oracle import nvfp4 as F4
from oracle import paged_attention as PA

# OCP MX v1.0, FP4 (E2M1) element values, codes 0..7 (sign bit clear)
OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_value_set_matches_ocp_table():
    assert list(e2m1.DECODE_TABLE[:8]) == OCP_E2M1
    assert list(e2m1.DECODE_TABLE[8:]) == [-v for v in OCP_E2M1]
    assert e2m1.E2M1_MAX == max(OCP_E2M1)


def test_grid_values_round_trip():
    for c in range(16):
        assert e2m1.encode(e2m1.DECODE_TABLE[c]) == c


@pytest.mark.parametrize("y,code", [
    (0.25, 0x0),   # between 0 (m=0) and 0.5 (m=1)
    (0.75, 0x2),   # between 0.5 (m=1) and 1.0 (m=0)
    (1.25, 0x2),   # between 1.0 (m=0) and 1.5 (m=1)
    (1.75, 0x4),   # between 1.5 (m=1) and 2.0 (m=0)
    (2.5, 0x4),    # between 2 (m=0) and 3 (m=1)
    (3.5, 0x6),    # between 3 (m=1) and 4 (m=0)
    (5.0, 0x6),    # between 4 (m=0) and 6 (m=1)
    (-2.5, 0xC), (-5.0, 0xE),
])
def test_midpoints_go_to_even_mantissa(y, code):
    assert e2m1.encode(y) == code


def test_saturation_nan_and_signed_zero():
    assert list(e2m1.encode([6.5, 100.0, np.inf, -np.inf, np.nan])) == [7, 7, 7, 15, 7]
    assert e2m1.encode(-0.1) == 0x8 and e2m1.encode(0.1) == 0x0


def test_nearest_by_brute_force():
    g = np.random.default_rng(1)
    y = np.concatenate([g.uniform(-8, 8, 20000),
                        np.array(OCP_E2M1)[1:] - 1e-6, np.array(OCP_E2M1)[:-1] + 1e-6])
    codes = e2m1.encode(y)
    grid = np.array(OCP_E2M1)
    for v, c in zip(y, codes):
        a = min(abs(v), 6.0)
        dist = np.abs(grid - a)
        best = np.flatnonzero(dist == dist.min())
        if len(best) == 2:       # tie: the even code
            best = [b for b in best if b % 2 == 0]
        assert (c & 7) == best[0], (v, c)
        assert (c >> 3) == (1 if v < 0 else 0)


def test_hand_worked_group():
    x = (0.75 * np.arange(16)).astype(np.float32)
    codes, sf = F4.quantize_row(x, 1.0)
    assert list(sf) == [0x3F]
    assert e4m3.decode(np.uint8(0x3F)) == 1.875
    # y = 0.4 i: 0, .4, .8, 1.2, 1.6, 2, 2.4, 2.8, 3.2, 3.6, 4, 4.4, 4.8, 5.2, 5.6, 6
    assert list(codes) == [0, 1, 2, 2, 3, 4, 4, 5, 5, 6, 6, 6, 6, 7, 7, 7]


def test_zero_tiny_and_huge_groups():
    z = np.zeros(32, np.float32)
    c, s = F4.quantize_row(z, 0.5)
    assert not c.any() and not s.any()
    # a / (6 S) below half the smallest E4M3 subnormal (2^-9): scale code 0
    tiny = np.full(16, 2.0 ** -12, np.float32)
    c, s = F4.quantize_row(tiny, 1.0)
    assert s[0] == 0 and not c.any()
    # a / (6 S) far above 448: the scale saturates to 448 (0x7E), the
    # elements to +-6
    big = np.array([1e6] + [-1e6] + [0.0] * 14, np.float32)
    c, s = F4.quantize_row(big, 1.0)
    assert s[0] == 0x7E and c[0] == 7 and c[1] == 15


def test_error_bound_random():
    g = np.random.default_rng(2)
    x = (g.standard_normal((64, 128)) * np.exp(g.uniform(-4, 4, (64, 1)))).astype(np.float32)
    S = float(np.abs(x).max()) / (6 * 448)
    c, s = F4.quantize_row(x, S)
    xh = np.stack([F4.dequantize_row(c[i], s[i], S) for i in range(64)])
    step = np.repeat(e4m3.decode(s), 16, axis=-1) * np.float32(S)
    # the grid spacing is at most 2 (between 4 and 6): half a step is 1
    assert np.all(np.abs(xh - x) <= step * 1.0 + 1e-30)
    # the group maximum is kept to within the E4M3 block-scale rounding
    gm = np.abs(x.reshape(64, 8, 16)).max(-1)
    ghm = np.abs(xh.reshape(64, 8, 16)).max(-1)
    assert np.all(np.abs(ghm - gm) <= gm * 0.25)


def _representable(g, shape, S):
    """Values code * 2^k * S with a +-6 element in every 16-group."""
    codes = g.integers(0, 16, shape).astype(np.uint8)
    codes[..., ::16] = np.where(g.random(codes[..., ::16].shape) < 0.5, 7, 15)
    k = g.integers(-6, 6, shape[:-1] + (shape[-1] // 16,))
    sc = np.repeat(2.0 ** k, 16, axis=-1)
    return (e2m1.decode(codes) * sc * S).astype(np.float32), codes, k


def test_lossless_round_trip():
    g = np.random.default_rng(3)
    S = 2.0 ** -3
    x, codes, k = _representable(g, (40, 128), S)
    c, s = F4.quantize_row(x, S)
    # -0 codes (0x8) come back as +0: same value
    assert np.array_equal(e2m1.decode(c), e2m1.decode(codes))
    assert np.array_equal(e4m3.decode(s), 2.0 ** k)


def test_layout_hand_packed():
    cache = F4.empty_cache(2, 1, 16, 32)
    S = 1.0
    # token rows whose codes are known: x = code value (scale 1 via a 6 in
    # each group)
    k0 = np.array([e2m1.DECODE_TABLE[c] for c in [1, 2] + [0] * 13 + [7]] * 2, np.float32)
    v2 = np.array([e2m1.DECODE_TABLE[c] for c in [3] + [0] * 14 + [7]] * 2, np.float32)
    v3 = np.array([e2m1.DECODE_TABLE[c] for c in [5] + [0] * 14 + [7]] * 2, np.float32)
    kn = np.stack([k0, k0, k0])[:, None, :]
    vn = np.stack([v2, v2, v3])[:, None, :]
    # tokens to block 1 offset 5 (K check), offsets 2 and 3 (V pair-row 1)
    k, ksf, v, vsf = F4.cache_write(kn, vn, [16 + 5, 16 + 2, 16 + 3], cache, S, S)
    assert k[1, 0, 5, 0] == 0x21                    # codes 1 (low), 2 (high)
    assert k[1, 0, 5, 7] == 0x70                    # codes 0, 7
    assert ksf[1, 0, 5, 0] == 0x38 and ksf[1, 0, 5, 1] == 0x38   # E4M3 1.0
    assert v[1, 0, 1, 0] == 0x53                    # token 2 low (3), 3 high (5)
    assert v[1, 0, 1, 15] == 0x77
    assert vsf[1, 0, 0, 2] == 0x38 and vsf[1, 0, 1, 3] == 0x38
    assert not k[0].any() and not v[0].any()


def test_decode_equals_dense_attention_on_representable_cache():
    g = np.random.default_rng(4)
    nb, hkv, bs, D, G = 12, 2, 16, 64, 4
    Sk, Sv = 2.0 ** -4, 2.0 ** -2
    lens = np.array([1, 17, 40, 0, 33])
    B = len(lens)
    perm = g.permutation(nb)
    tables = np.full((B, 3), -1)
    u = 0
    for b, n in enumerate(lens):
        for j in range(-(-n // bs)):
            tables[b, j] = perm[u % nb]
            u += 1
    T = nb * bs
    kx, _, _ = _representable(g, (T, hkv, D), Sk)
    vx, _, _ = _representable(g, (T, hkv, D), Sv)
    cache = F4.cache_write(kx, vx, np.arange(T), F4.empty_cache(nb, hkv, bs, D), Sk, Sv)
    # the same values as a dense float cache [nb, hkv, bs, D]
    kd = kx.reshape(nb, bs, hkv, D).transpose(0, 2, 1, 3)
    vd = vx.reshape(nb, bs, hkv, D).transpose(0, 2, 1, 3)
    q = g.standard_normal((B, hkv * G, D))
    ref = PA.decode(q, kd, vd, tables, lens, 0.125)
    got = F4.decode(q, cache, Sk, Sv, tables, lens, 0.125)
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_pages_nvfp4_footprint():
    # 2 * 80 layers * 8 KV heads * 128 * 131072 tokens at 4 bits per value
    bits4 = footprint.kv_bytes_per_token(80, 8, 128, 1) * 131072 // 2
    assert round(bits4 / 1e9, 1) == 10.7
    assert bits4 * 4 == footprint.kv_bytes_per_token(80, 8, 128, 2) * 131072
    # with one E4M3 block scale per 16 values: 4.5 bits per value
    with_sf = footprint.nvfp4_bytes_per_token(80, 8, 128) * 131072
    assert with_sf == bits4 * 9 // 8
