"""Per-(block, KV head) absmax FP8 E4M3 quantisation (oracle; test only).

The page "Paged Attention and KV Cache Fragmentation", section "Quantization
as a way to stretch paged memory further", motivates FP8 KV caches (half the
BF16 footprint) and warns that accumulation must stay in full fp32.  It fixes
neither the scale granularity nor the rounding; this restatement takes the
plainest reading, one fp32 scale per (physical block, KV head), separately for
K and V:

    a      = max |x|  over the block's valid tokens and the head dimension
    scale  = a / 448            (fp32 IEEE division; 1.0 when a == 0)
    code   = e4m3_rne_satfinite(x / scale)   (fp32 IEEE division per element)

Slots at or beyond the block's valid length are written as code 0 (+0.0).
Dequantised value = decode(code) * scale.
"""
from __future__ import annotations

import numpy as np

from . import e4m3


def block_scale(x_block_f32: np.ndarray) -> np.float32:
    """Scale of one (block, head) tile: fp32 absmax / 448, or 1 when all zero."""
    a = np.float32(np.max(np.abs(x_block_f32))) if x_block_f32.size else np.float32(0)
    if a == 0:
        return np.float32(1.0)
    return np.float32(a) / np.float32(e4m3.E4M3_MAX)


def quantize_tile(x_tile_f32: np.ndarray, valid: int):
    """Quantise one [block_size, d] tile; returns (uint8 codes, fp32 scale)."""
    x = np.asarray(x_tile_f32, dtype=np.float32)
    codes = np.zeros(x.shape, dtype=np.uint8)
    s = block_scale(x[:valid])
    if valid > 0:
        q = (x[:valid] / s).astype(np.float32)     # fp32 IEEE divide
        codes[:valid] = e4m3.encode_fast(q)
    return codes, s


def quantize_blocks(cache_f32: np.ndarray, block_ids, valid_lens):
    """Quantise listed blocks of a [num_blocks, Hkv, bs, d] cache.

    Returns (codes uint8 [num_blocks, Hkv, bs, d], scales fp32 [num_blocks,
    Hkv]).  Blocks not listed keep code 0 and scale 1.
    """
    nb, hkv, bs, d = cache_f32.shape
    codes = np.zeros((nb, hkv, bs, d), dtype=np.uint8)
    scales = np.ones((nb, hkv), dtype=np.float32)
    block_ids = np.asarray(block_ids, dtype=np.int64)
    valid_lens = np.asarray(valid_lens, dtype=np.int64)
    # Whole blocks: the same arithmetic as quantize_tile, batched over
    # blocks and heads (one absmax per (block, head), one divide per value).
    full = block_ids[valid_lens == bs]
    if full.size:
        x = np.asarray(cache_f32[full], dtype=np.float32)
        a = np.max(np.abs(x), axis=(2, 3)).astype(np.float32)
        s = np.where(a == 0, np.float32(1.0),
                     a / np.float32(e4m3.E4M3_MAX)).astype(np.float32)
        codes[full] = e4m3.encode_fast((x / s[:, :, None, None]).astype(np.float32))
        scales[full] = s
    for blk, valid in zip(block_ids, valid_lens):
        if valid == bs:
            continue
        for h in range(hkv):
            c, s = quantize_tile(cache_f32[blk, h], int(valid))
            codes[blk, h] = c
            scales[blk, h] = s
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """fp64 values decode(code) * scale for a whole [nb, Hkv, bs, d] cache."""
    return e4m3.decode(codes) * scales.astype(np.float64)[:, :, None, None]


# ------------------------------------------------------------ FP8 append ---
# Appending a token to an FP8 block.  The pages name only whole-block
# quantisation; appending into a partly filled block is this restatement's
# reading, the plainest one that keeps one fp32 scale per (block, KV head)
# and never lets a stored value overflow:
#
#   the token's own scale   s_t = a_t / 448        (a_t = max |x_t|; fp32)
#   first token of a block  (offset 0): scale = s_t, or 1 when a_t == 0
#   later tokens            scale = max(old scale, s_t)   ("grow only")
#   when the scale grows, every earlier row r < offset is requantised:
#       y    = decode(code) * old_scale          (fp32 product, RN)
#       code = e4m3_rne_satfinite(y / new_scale) (fp32 IEEE divide)
#   the token itself        code = e4m3_rne_satfinite(x_t / scale)
#
# Filling a block in order of falling absmax therefore never requantises and
# gives exactly the whole-block quantiser's codes, and whatever the order the
# final scale equals the whole-block scale of the block's tokens.


def append_token(codes_tile: np.ndarray, scale, offset: int, x_f32: np.ndarray):
    """Append one token row x (fp32 [d]) at ``offset`` of one (block, head)
    tile of codes (uint8 [bs, d], rows >= offset unused).  Returns the new
    (codes, scale); the input is not modified."""
    codes = np.array(codes_tile, dtype=np.uint8, copy=True)
    x = np.asarray(x_f32, dtype=np.float32)
    a = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    s_t = np.float32(a / np.float32(e4m3.E4M3_MAX))
    old = np.float32(scale)
    if offset == 0:
        new = np.float32(1.0) if a == 0 else s_t
    elif s_t > old:
        new = s_t
        y = (e4m3.decode(codes[:offset]).astype(np.float32) * old).astype(np.float32)
        codes[:offset] = e4m3.encode_fast((y / new).astype(np.float32))
    else:
        new = old
    codes[offset] = e4m3.encode_fast((x / new).astype(np.float32))
    return codes, new


def cache_write_fp8(k_new, v_new, slots, k_codes, v_codes, k_scale, v_scale):
    """FP8 cache write of tokens t (in order) with slot s = slots[t] >= 0:
    append_token on block s // bs, row s % bs, for every KV head, K and V.
    Arrays are copied; returns (k_codes, v_codes, k_scale, v_scale)."""
    kc, vc = np.array(k_codes, copy=True), np.array(v_codes, copy=True)
    ks, vs = np.array(k_scale, copy=True), np.array(v_scale, copy=True)
    bs = kc.shape[2]
    for t, s in enumerate(np.asarray(slots, dtype=np.int64)):
        if s < 0:
            continue
        blk, off = int(s) // bs, int(s) % bs
        for h in range(kc.shape[1]):
            kc[blk, h], ks[blk, h] = append_token(kc[blk, h], ks[blk, h], off, k_new[t, h])
            vc[blk, h], vs[blk, h] = append_token(vc[blk, h], vs[blk, h], off, v_new[t, h])
    return kc, vc, ks, vs
