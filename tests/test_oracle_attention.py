"""Pins for the oracle's paged decode attention, cache write and block copy.

Each test pins the oracle to something other than itself:
* closed forms: a hand-worked two-token case, seq_len = 1 -> V, identical
  keys -> mean(V), scale = 0 -> mean(V), one dominant key -> its V row;
* brute force: a pure-Python gather (explicit loops over tokens) fed to
  torch's fp64 scaled_dot_product_attention;
* invariants: permuting physical block ids (data moved with the table) and
  shared-vs-copied prefix blocks leave the output bit-identical;
* GQA grouping: query head h reads KV head h // G (the h % Hkv mapping is
  shown to give a different answer, so a swapped index would be caught);
* numerics: scores of magnitude ~1e3 stay finite (max subtraction present).
"""
import math

import numpy as np
import pytest
import torch

from oracle import paged_attention as PA
from oracle import quantize as QZ


def _rand_case(seed, B=3, Hq=4, Hkv=2, d=8, bs=4, lens=(1, 5, 11), nb=16):
    g = np.random.default_rng(seed)
    k = g.standard_normal((nb, Hkv, bs, d))
    v = g.standard_normal((nb, Hkv, bs, d))
    q = g.standard_normal((B, Hq, d))
    perm = g.permutation(nb)
    maxb = max(-(-n // bs) for n in lens)
    tables = -np.ones((B, maxb), dtype=np.int64)
    i = 0
    for b, n in enumerate(lens):
        for j in range(-(-n // bs)):
            tables[b, j] = perm[i]
            i += 1
    return q, k, v, tables, np.array(lens), bs


def test_hand_worked_two_tokens():
    # q = [1, 0]; keys [1, 0], [0, 1]; values [1, 2], [3, 4]; scale 1:
    # weights e^1 : e^0, out = (e*[1,2] + [3,4]) / (e + 1)
    q = np.array([[[1.0, 0.0]]])
    k = np.zeros((1, 1, 2, 2))
    v = np.zeros((1, 1, 2, 2))
    k[0, 0] = [[1, 0], [0, 1]]
    v[0, 0] = [[1, 2], [3, 4]]
    out = PA.decode(q, k, v, np.array([[0]]), np.array([2]), 1.0)
    e = math.e
    np.testing.assert_allclose(out[0, 0], [(e + 3) / (e + 1), (2 * e + 4) / (e + 1)],
                               rtol=0, atol=1e-15)
    # the scale multiplies the scores: scale 2 gives weights e^2 : 1
    out2 = PA.decode(q, k, v, np.array([[0]]), np.array([2]), 2.0)
    e2 = math.e ** 2
    np.testing.assert_allclose(out2[0, 0], [(e2 + 3) / (e2 + 1), (2 * e2 + 4) / (e2 + 1)],
                               rtol=0, atol=1e-15)


def test_seq_len_one_returns_v_exactly():
    q, k, v, t, _, bs = _rand_case(1)
    out = PA.decode(q, k, v, t, np.array([1, 1, 1]), 0.7)
    for b in range(3):
        for h in range(4):
            assert np.array_equal(out[b, h], v[t[b, 0], h // 2, 0])


def test_identical_keys_and_zero_scale_give_mean_of_v():
    q, k, v, t, lens, bs = _rand_case(2)
    k_same = np.broadcast_to(k[:1, :, :1, :], k.shape).copy()
    for kk, sc in ((k_same, 0.9), (k, 0.0)):
        out = PA.decode(q, kk, v, t, lens, sc)
        for b in range(3):
            for h in range(4):
                rows = [v[t[b, i // bs], h // 2, i % bs] for i in range(lens[b])]
                np.testing.assert_allclose(out[b, h], np.mean(rows, axis=0),
                                           rtol=1e-13, atol=1e-13)


def test_dominant_key_selects_its_value():
    q, k, v, t, lens, bs = _rand_case(3)
    b, h, pos = 2, 1, 6
    kv = h // 2
    k = k.copy()
    k[t[b, pos // bs], kv, pos % bs] = 100.0 * q[b, h] / np.linalg.norm(q[b, h])
    out = PA.decode(q, k, v, t, lens, 1.0)
    np.testing.assert_allclose(out[b, h], v[t[b, pos // bs], kv, pos % bs],
                               rtol=0, atol=1e-12)


def _python_gather(cache, row, n, bs):
    keys = []
    for tok in range(n):
        blk = int(row[tok // bs])
        keys.append([float(x) for x in cache[blk, :, tok % bs, :].reshape(-1)])
    return keys


@pytest.mark.parametrize("seed", [4, 5, 6])
def test_brute_force_against_torch_sdpa(seed):
    q, k, v, t, lens, bs = _rand_case(seed, B=3, Hq=6, Hkv=2, d=8, bs=4,
                                      lens=(3, 9, 16), nb=20)
    sc = 0.37
    out = PA.decode(q, k, v, t, lens, sc)
    G = 3
    for b in range(3):
        kk = np.array(_python_gather(k, t[b], lens[b], bs)).reshape(lens[b], 2, 8)
        vv = np.array(_python_gather(v, t[b], lens[b], bs)).reshape(lens[b], 2, 8)
        for h in range(6):
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q[b, h][None, None, None, :]),
                torch.tensor(kk[None, None, :, h // G, :]),
                torch.tensor(vv[None, None, :, h // G, :]), scale=sc)
            np.testing.assert_allclose(out[b, h], ref.numpy().reshape(-1),
                                       rtol=1e-12, atol=1e-12)


def test_gqa_grouping_is_h_div_g():
    q, k, v, t, lens, bs = _rand_case(8, B=1, Hq=4, Hkv=2, d=8, bs=4,
                                      lens=(10,), nb=6)
    out = PA.decode(q, k, v, t, lens, 0.5)
    for h in range(4):
        ref = PA.attend(q[0, h], PA.gather_sequence(k, t[0], 10, bs)[:, h // 2],
                        PA.gather_sequence(v, t[0], 10, bs)[:, h // 2], 0.5)
        wrong = PA.attend(q[0, h], PA.gather_sequence(k, t[0], 10, bs)[:, h % 2],
                          PA.gather_sequence(v, t[0], 10, bs)[:, h % 2], 0.5)
        assert np.array_equal(out[0, h], ref)
        if h in (1, 2):
            assert not np.allclose(ref, wrong)


def test_physical_permutation_invariance_is_bit_exact():
    q, k, v, t, lens, bs = _rand_case(9, nb=16)
    out = PA.decode(q, k, v, t, lens, 0.8)
    perm = np.random.default_rng(99).permutation(16)   # new id of block i
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    t2 = np.where(t >= 0, perm[np.maximum(t, 0)], -1)
    out2 = PA.decode(q, k2, v2, t2, lens, 0.8)
    assert np.array_equal(out, out2)


def test_shared_vs_copied_prefix_is_bit_exact():
    g = np.random.default_rng(10)
    bs, d = 4, 8
    k = g.standard_normal((12, 1, bs, d))
    v = g.standard_normal((12, 1, bs, d))
    q = g.standard_normal((2, 1, d))
    shared = np.array([[0, 1, 2], [0, 1, 3]])
    out_s = PA.decode(q, k, v, shared, np.array([11, 12]), 0.3)
    k[5], v[5] = k[0], v[0]
    k[6], v[6] = k[1], v[1]
    copied = np.array([[0, 1, 2], [5, 6, 3]])
    out_c = PA.decode(q, k, v, copied, np.array([11, 12]), 0.3)
    assert np.array_equal(out_s, out_c)


def test_large_scores_stay_finite():
    q, k, v, t, lens, bs = _rand_case(11)
    out = PA.decode(q * 300.0, k, v, t, lens, 1.0)
    assert np.all(np.isfinite(out))


def test_empty_sequence_gives_zeros():
    q, k, v, t, lens, bs = _rand_case(12)
    out = PA.decode(q, k, v, t, np.array([0, 5, 11]), 1.0)
    assert np.array_equal(out[0], np.zeros_like(out[0]))


def test_table_entries_past_length_are_never_read():
    q, k, v, t, lens, bs = _rand_case(13, lens=(5, 5, 5), nb=16)
    t = np.concatenate([t, np.full((3, 4), 10 ** 9)], axis=1)
    out = PA.decode(q, k, v, t, lens, 1.0)
    assert np.all(np.isfinite(out))


def test_cache_write_matches_elementwise_loop():
    g = np.random.default_rng(14)
    nb, H, bs, d, T = 6, 2, 4, 3, 7
    kc = g.integers(0, 2 ** 16, (nb, H, bs, d), dtype=np.uint16)
    vc = g.integers(0, 2 ** 16, (nb, H, bs, d), dtype=np.uint16)
    kn = g.integers(0, 2 ** 16, (T, H, d), dtype=np.uint16)
    vn = g.integers(0, 2 ** 16, (T, H, d), dtype=np.uint16)
    slots = np.array([3, -1, 17, 0, 23, -5, 9])
    k2, v2 = PA.cache_write(kn, vn, slots, kc, vc)
    ek, ev = kc.copy(), vc.copy()
    for tok in range(T):
        s = int(slots[tok])
        if s < 0:
            continue
        for h in range(H):
            for i in range(d):
                ek[s // bs, h, s % bs, i] = kn[tok, h, i]
                ev[s // bs, h, s % bs, i] = vn[tok, h, i]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)
    assert np.array_equal(kc[1], k2[1])  # untouched block unchanged


def test_copy_blocks_copies_prefix_only():
    g = np.random.default_rng(15)
    kc = g.integers(0, 255, (5, 2, 4, 3), dtype=np.uint8)
    vc = g.integers(0, 255, (5, 2, 4, 3), dtype=np.uint8)
    k2, v2 = PA.copy_blocks(kc, vc, [(1, 3, 2), (0, 4, 4)])
    assert np.array_equal(k2[3, :, :2], kc[1, :, :2])
    assert np.array_equal(k2[3, :, 2:], kc[3, :, 2:])
    assert np.array_equal(v2[4], vc[0])
    assert np.array_equal(k2[:3], kc[:3])


def test_fp8_decode_equals_float_decode_on_dequantised_cache():
    q, k, v, t, lens, bs = _rand_case(16, nb=16)
    k32, v32 = k.astype(np.float32), v.astype(np.float32)
    used = sorted({int(x) for x in t.ravel() if x >= 0})
    kq, ks = QZ.quantize_blocks(k32, used, [bs] * len(used))
    vq, vs = QZ.quantize_blocks(v32, used, [bs] * len(used))
    a = PA.decode(q, kq, vq, t, lens, 0.6, k_scale=ks, v_scale=vs)
    b = PA.decode(q, QZ.dequantize(kq, ks), QZ.dequantize(vq, vs), t, lens, 0.6)
    assert np.array_equal(a, b)
