"""NVFP4 KV cache: two-level scaled FP4 quantisation, layout, decode (oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The page "Paged Attention and KV Cache Fragmentation", section "Quantization
as a way to stretch paged memory further", names NVFP4 as the Blackwell-only
KV format that halves FP8 again, and leaves the format itself undefined.  The
plainest reading is NVIDIA's published NVFP4 (the FP4 E2M1 element of the OCP
MX specification with a finer block scale and a second, per-tensor scale):

    16 consecutive elements along the head dimension share one E4M3 scale;
    one fp32 scale S per tensor (here: the K cache, resp. V cache, of one
    layer) brings those block scales into E4M3's range.

Quantisation of one token row x (fp32, the bf16 input widened exactly), with
every step in fp32 IEEE arithmetic (round to nearest even), the precision
the CUDA kernel decides the codes in:

    a_g  = max |x_i| over group g (16 elements)
    s_g  = e4m3_rne_satfinite(a_g / (6 * S))      # block scale, an E4M3 code
    q_i  = e2m1_rne_satfinite(x_i / (dec(s_g) * S))  if dec(s_g) > 0, else +0

Dequantised value: e2m1(q_i) * e4m3(s_g) * S.  S is the caller's calibration
(for example amax / (6 * 448) over the tensor); it must be positive and
finite.

Cache layout per (block, KV head), block_size tokens (a multiple of 16) and
head dimension D, all uint8 -- a choice of this library, not of the pages
(see the kernels' description):

    k      [bs][D/2]       byte j of token t = q(t, 2j) | q(t, 2j+1) << 4
    k_sf   [bs][D/16]      E4M3 block scale of group g of token t
    v      [bs/2][D]       byte d of pair-row p = q(2p, d) | q(2p+1, d) << 4
    v_sf   [D/16][bs]      E4M3 block scale of group g of token t (group-major)

so the whole caches are k [num_blocks, Hkv, bs, D/2], k_sf [num_blocks, Hkv,
bs, D/16], v [num_blocks, Hkv, bs/2, D], v_sf [num_blocks, Hkv, D/16, bs].
"""
from __future__ import annotations

import numpy as np

from . import e2m1, e4m3
from .paged_attention import attend

GROUP = 16


# ------------------------------------------------------------- quantise ---
def quantize_row(x_f32, S):
    """Quantise rows (fp32 [..., D], D a multiple of 16) with tensor scale S.

    Returns (codes uint8 [..., D], one 4-bit code per element; block scales
    uint8 [..., D/16], E4M3 codes)."""
    x = np.asarray(x_f32, dtype=np.float32)
    S = np.float32(S)
    g = x.reshape(x.shape[:-1] + (-1, GROUP))
    a = np.max(np.abs(g), axis=-1).astype(np.float32)
    d6 = np.float32(np.float32(6.0) * S)
    sf = e4m3.encode_fast((a / d6).astype(np.float32))
    sv = e4m3.decode(sf).astype(np.float32)          # exact
    den = (sv * S).astype(np.float32)
    codes = np.zeros(g.shape, dtype=np.uint8)
    nz = sv > 0
    if np.any(nz):
        y = (g[nz] / den[nz][:, None]).astype(np.float32)
        codes[nz] = e2m1.encode(y)
    return codes.reshape(x.shape), sf


def dequantize_row(codes, sf, S) -> np.ndarray:
    """fp64 values e2m1(code) * e4m3(scale of its group) * S of one row."""
    c = np.asarray(codes, dtype=np.uint8)
    s = e4m3.decode(np.asarray(sf, dtype=np.uint8))
    return e2m1.decode(c) * np.repeat(s, GROUP) * float(np.float32(S))


# --------------------------------------------------------------- layout ---
def empty_cache(num_blocks, num_kv_heads, block_size, head_dim):
    """Zero-filled (k, k_sf, v, v_sf) arrays in the layout above."""
    nb, h, bs, d = num_blocks, num_kv_heads, block_size, head_dim
    return (np.zeros((nb, h, bs, d // 2), np.uint8), np.zeros((nb, h, bs, d // 16), np.uint8),
            np.zeros((nb, h, bs // 2, d), np.uint8), np.zeros((nb, h, d // 16, bs), np.uint8))


def cache_write(k_new, v_new, slots, cache, k_gs, v_gs):
    """Quantise and store tokens t with slot s = slots[t] >= 0 at block
    s // bs, offset s % bs, every KV head.  ``k_new``/``v_new`` are fp32
    [T, Hkv, D] (bf16 inputs widened); ``cache`` is (k, k_sf, v, v_sf).
    Slots must be distinct.  Returns updated copies."""
    k, k_sf, v, v_sf = (np.array(a, copy=True) for a in cache)
    bs = k.shape[2]
    slots = np.asarray(slots, dtype=np.int64)
    keep = slots >= 0
    s = slots[keep]
    blk, off = s // bs, s % bs
    kc, kf = quantize_row(np.asarray(k_new, np.float32)[keep], k_gs)   # [n, Hkv, D]
    vc, vf = quantize_row(np.asarray(v_new, np.float32)[keep], v_gs)
    k[blk, :, off] = kc[..., 0::2] | (kc[..., 1::2] << 4)
    k_sf[blk, :, off] = kf
    # V: token 2p in the low nibbles of pair-row p, token 2p + 1 in the high
    for hi in (0, 1):
        m = off % 2 == hi
        b, p = blk[m], off[m] // 2
        row = v[b, :, p]
        v[b, :, p] = ((row & 0x0F) | (vc[m] << 4)) if hi else ((row & 0xF0) | vc[m])
    v_sf[blk, :, :, off] = vf
    return k, k_sf, v, v_sf


def gather_rows(cache, k_gs, v_gs, table_row, n, h):
    """Dequantised fp64 K and V rows [n, D] of one sequence's KV head h:
    token t is read from block table_row[t // bs] at offset t % bs, its K
    codes from both nibbles of its row, its V codes from the low (even t) or
    high (odd t) nibbles of pair-row (t % bs) // 2, each value times its
    group's E4M3 scale and the tensor scale."""
    k, k_sf, v, v_sf = cache
    bs, D = k.shape[2], v.shape[3]
    t = np.arange(int(n))
    blk = np.asarray(table_row, dtype=np.int64)[t // bs]
    off = t % bs
    kb = k[blk, h, off]                                      # [n, D/2]
    kc = np.stack([kb & 0xF, kb >> 4], axis=-1).reshape(len(t), D)
    ks = np.repeat(e4m3.decode(k_sf[blk, h, off]), GROUP, axis=-1)
    vb = v[blk, h, off // 2]                                 # [n, D]
    vc = np.where((off % 2 == 1)[:, None], vb >> 4, vb & 0xF)
    vs = np.repeat(e4m3.decode(v_sf[blk, h, :, off]), GROUP, axis=-1)
    K = e2m1.decode(kc) * ks * float(np.float32(k_gs))
    V = e2m1.decode(vc) * vs * float(np.float32(v_gs))
    return K, V


# --------------------------------------------------------------- decode ---
def decode(q, cache, k_gs, v_gs, block_tables, seq_lens, scale, *, seqs=None,
           heads=None):
    """Paged decode attention over an NVFP4 cache, fp64: each sequence's K/V
    rows are gathered through its block table and dequantised, then
    softmax(scale * q . k) . v per query head (KV head h // G).  ``seqs`` /
    ``heads`` restrict the outputs computed; the others stay NaN."""
    q = np.asarray(q)
    B, Hq, D = q.shape
    Hkv = cache[0].shape[1]
    G = Hq // Hkv
    out = np.full((B, Hq, D), np.nan)
    for b in (range(B) if seqs is None else seqs):
        n = int(seq_lens[b])
        hs = list(range(Hq) if heads is None else heads)
        for g in sorted({h // G for h in hs}):
            K, V = gather_rows(cache, k_gs, v_gs, block_tables[b], n, g)
            for h in hs:
                if h // G == g:
                    out[b, h] = attend(q[b, h], K, V, scale)
    return out
