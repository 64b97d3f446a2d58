"""Paged KV cache: scatter write, block copy and decode attention (oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the pages fix
------------------
* "KV cache fragmentation" (field guide), section "Definition": the cache is
  cut into small fixed-size pages; each request owns a logical sequence of
  pages scattered anywhere in physical memory, with an indirection table from
  logical position to physical page, and the attention kernel walks it.
* "Paged Attention and KV Cache Fragmentation", section "How PagedAttention
  maps an OS concept onto GPU memory": every block holds a fixed number of
  key/value vectors per attention head; a request sees its cache as one
  continuous sequence while the blocks may sit anywhere; blocks are allocated
  only as a sequence grows; requests sharing a prefix point at the same
  physical block.

So paged decode reaches exactly (up to rounding order) dense attention over
the logically contiguous sequence.  This module writes that definition out:
gather through the block table into contiguous fp64 arrays, then
softmax(scale * q . k) . v per query head, with grouped-query heads mapped to
KV head ``h // G`` (contiguous groups; the pages only name GQA, in the lesson
navigation of the "Fragmentation" page).  The attention formula is the
textbook scaled dot-product attention (Vaswani et al. 2017, eq. 1) for one
query row.

Layouts (all plain numpy arrays):
    k_cache, v_cache : [num_blocks, Hkv, block_size, d]
    block_tables     : int [B, max_blocks]  (entries past a sequence's last
                       block are never read)
    seq_lens         : int [B]  (length after this step's append)
    q                : [B, Hq, d];  out : float64 [B, Hq, d]
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------- gather ---
def gather_sequence(cache: np.ndarray, table_row: np.ndarray, seq_len: int,
                    block_size: int) -> np.ndarray:
    """Contiguous [seq_len, Hkv, d] view of one sequence's cache.

    Logical token t lives in physical block ``table_row[t // block_size]`` at
    offset ``t % block_size`` (the page-table mapping of the pages above).
    """
    t = np.arange(int(seq_len))
    blk = np.asarray(table_row)[t // block_size]
    off = t % block_size
    return cache[blk, :, off, :]


# ----------------------------------------------------------------- attend ---
def attend(q_row: np.ndarray, keys: np.ndarray, values: np.ndarray,
           scale: float) -> np.ndarray:
    """softmax(scale * keys @ q) @ values for one query vector, in fp64.

    An empty key set returns zeros (a sequence of length 0 attends to nothing;
    the pages are silent, this is the reading the library also implements).
    """
    q64 = np.asarray(q_row, dtype=np.float64)
    k64 = np.asarray(keys, dtype=np.float64)
    v64 = np.asarray(values, dtype=np.float64)
    if k64.shape[0] == 0:
        return np.zeros(v64.shape[-1], dtype=np.float64)
    s = float(scale) * (k64 @ q64)
    m = np.max(s)
    p = np.exp(s - m)
    return (p @ v64) / np.sum(p)


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale, *,
           num_kv_heads=None, k_scale=None, v_scale=None,
           seqs=None, heads=None):
    """Paged single-token decode attention, fp64.

    ``k_cache``/``v_cache`` hold values (any float dtype) or, when
    ``k_scale``/``v_scale`` (fp32 [num_blocks, Hkv]) are given, E4M3 codes
    (uint8) that dequantise to decode(code) * scale of their (block, head).
    ``seqs``/``heads`` restrict the computation to a subset of (sequence,
    query head) outputs (for sampled checks of large workloads); other entries
    of the returned array stay NaN.
    """
    q = np.asarray(q)
    B, Hq, d = q.shape
    Hkv = k_cache.shape[1] if num_kv_heads is None else num_kv_heads
    G = Hq // Hkv
    bs = k_cache.shape[2]
    out = np.full((B, Hq, d), np.nan, dtype=np.float64)
    seqs = range(B) if seqs is None else seqs
    for b in seqs:
        n = int(seq_lens[b])
        hs = range(Hq) if heads is None else heads
        groups = sorted({h // G for h in hs})
        for g in groups:
            kc = gather_sequence(k_cache[:, g:g + 1], block_tables[b], n, bs)[:, 0]
            vc = gather_sequence(v_cache[:, g:g + 1], block_tables[b], n, bs)[:, 0]
            if k_scale is not None:
                t = np.arange(n)
                blk = np.asarray(block_tables[b])[t // bs]
                kc = dequant_rows(kc, k_scale[blk, g])
                vc = dequant_rows(vc, v_scale[blk, g])
            for h in hs:
                if h // G != g:
                    continue
                out[b, h] = attend(q[b, h], kc, vc, scale)
    return out


def dequant_rows(codes_rows: np.ndarray, row_scales: np.ndarray) -> np.ndarray:
    """fp64 decode(code) * scale for gathered rows [n, d] with scales [n]."""
    from . import e4m3
    return e4m3.decode(codes_rows) * np.asarray(row_scales, np.float64)[:, None]


# ------------------------------------------------------------ cache write ---
def cache_write(k_new, v_new, slot_mapping, k_cache, v_cache):
    """Scatter each new token's K/V into its slot; returns updated copies.

    Slot s names physical block ``s // block_size`` and offset
    ``s % block_size``; a negative slot means "skip this token".  Values are
    copied bit for bit (any dtype, including raw uint16 / uint8 views).
    Duplicate slots are outside the contract; here the later token wins.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    bs = kc.shape[2]
    for t, s in enumerate(np.asarray(slot_mapping).tolist()):
        if s < 0:
            continue
        kc[s // bs, :, s % bs, :] = k_new[t]
        vc[s // bs, :, s % bs, :] = v_new[t]
    return kc, vc


# ------------------------------------------------------------ block copy ---
def copy_blocks(k_cache, v_cache, pairs):
    """Copy the first ``n`` slots of block ``src`` into block ``dst``.

    ``pairs`` rows are (src, dst, n); all heads, K and V, bit for bit.  This
    is the copy-on-write step for a shared partial block: sequences that share
    physical blocks diverge only where their content differs ("Paged Attention
    and KV Cache Fragmentation", section "How PagedAttention maps an OS concept
    onto GPU memory").  Pairs are applied in order.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    for src, dst, n in np.asarray(pairs).reshape(-1, 3).tolist():
        kc[dst, :, :n, :] = kc[src, :, :n, :]
        vc[dst, :, :n, :] = vc[src, :, :n, :]
    return kc, vc
