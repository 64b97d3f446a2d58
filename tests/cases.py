"""Test-side construction of paged decode cases and their oracle answers.

Inputs come from the seeded generators in ``paged_kv_cache_228_gb300.
workloads``; block tables and the append step's slots come from the oracle's
block-manager model.  Expected values come only from ``oracle/``: for each
checked sequence the blocks it uses are copied out of the generated pool
BEFORE any library kernel touches it, and the oracle applies the cache write
and the attention itself.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from oracle import block_manager as BM
from oracle import paged_attention as OPA
from oracle import quantize as OQ
from paged_kv_cache_228_gb300 import workloads as W


@dataclass
class Case:
    w: W.Workload
    device: str
    tables: list          # per-seq block ids after the append (python lists)
    pre_lens: list        # lengths before the append
    slots: list           # append slot per sequence
    cow_pairs: list
    k_cache: torch.Tensor  # bf16 pool, pre-write contents
    v_cache: torch.Tensor
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    table_t: torch.Tensor  # int32 [B, max_blocks] padded with -1
    lens_t: torch.Tensor   # int32 [B] post-append
    slots_t: torch.Tensor  # int64 [B]


def build_case(w: W.Workload, device="cuda", poison_unused=False, gen_device=None) -> Case:
    ops = W.build_script(w)
    maxb = w.max_blocks_per_seq
    model, tables, lens = BM.replay_script(ops, w.num_seqs, w.block_size, maxb, w.pool_blocks)
    slots, pairs = [], []
    for b in range(w.num_seqs):
        st, s, pr = model.append_slots(tables[b], lens[b], 1, w.block_size, maxb)
        assert st == BM.OK
        slots += s
        pairs += pr
    gd = gen_device or device
    shape = (w.pool_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    k = W.normal_bf16(shape, w.seed * 10 + 1, gd, w.outlier_prob, w.outlier_scale).to(device)
    v = W.normal_bf16(shape, w.seed * 10 + 2, gd, w.outlier_prob, w.outlier_scale).to(device)
    if poison_unused:
        used = torch.zeros(w.pool_blocks, dtype=torch.bool)
        for t in tables:
            used[t] = True
        k[~used.to(device)] = float("nan")
        v[~used.to(device)] = float("nan")
        # unused slots of the last block of each sequence
        for b, t in enumerate(tables):
            n = w.seq_lens[b]
            tail = n % w.block_size
            if tail:
                k[t[-1], :, tail:, :] = float("nan")
                v[t[-1], :, tail:, :] = float("nan")
    q = W.normal_bf16((w.num_seqs, w.num_q_heads, w.head_dim), w.seed * 10 + 3).to(device)
    kn = W.normal_bf16((w.num_seqs, w.num_kv_heads, w.head_dim), w.seed * 10 + 4).to(device)
    vn = W.normal_bf16((w.num_seqs, w.num_kv_heads, w.head_dim), w.seed * 10 + 5).to(device)
    tab = torch.full((w.num_seqs, maxb), -1, dtype=torch.int32)
    for b, t in enumerate(tables):
        tab[b, :len(t)] = torch.tensor(t, dtype=torch.int32)
    return Case(w, device, tables, lens, slots, pairs, k, v, q, kn, vn,
                tab.to(device), torch.tensor(w.seq_lens, dtype=torch.int32).to(device),
                torch.tensor(slots, dtype=torch.int64).to(device))


def _to_np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def _to_np32(t: torch.Tensor) -> np.ndarray:
    # bf16 -> fp32 is exact; the oracle widens to fp64 where it computes
    return t.detach().to("cpu").to(torch.float32).numpy()


def snapshot_blocks(case: Case, seqs):
    """Copy the pre-write blocks of ``seqs`` to host: (ids, k, v) where k/v
    are float32 [len(ids), Hkv, bs, d] holding the bf16 values exactly.
    Call before any library kernel touches the pool."""
    ids = sorted({bid for b in seqs for bid in case.tables[b]})
    idx = torch.tensor(ids, dtype=torch.int64, device=case.k_cache.device)
    return ids, _to_np32(case.k_cache.index_select(0, idx)), _to_np32(case.v_cache.index_select(0, idx))


def oracle_decode(case: Case, snap, seqs, heads=None, with_append=True, lens=None, scale=None):
    """fp64 oracle output [B, Hq, d] (NaN outside ``seqs``/``heads``).
    ``lens`` overrides the workload's post-append lengths, ``scale`` its
    softmax scale."""
    ids, kk, vv = snap
    local = {bid: i for i, bid in enumerate(ids)}
    bs = case.w.block_size
    seqs = list(seqs)
    maxb = max(len(t) for t in case.tables)
    tab = -np.ones((case.w.num_seqs, maxb), dtype=np.int64)
    for b in seqs:
        tab[b, :len(case.tables[b])] = [local[x] for x in case.tables[b]]
    if with_append:
        sl = np.full(case.w.num_seqs, -1, dtype=np.int64)
        for b in seqs:
            s = case.slots[b]
            sl[b] = local[s // bs] * bs + s % bs
        kk, vv = OPA.cache_write(_to_np32(case.k_new), _to_np32(case.v_new), sl, kk, vv)
    lens = np.array(case.w.seq_lens if lens is None else lens)
    return OPA.decode(_to_np64(case.q), kk, vv, tab, lens,
                      case.w.scale if scale is None else scale, seqs=seqs, heads=heads)


def oracle_decode_fp8(case: Case, snap, seqs, heads=None):
    """Oracle on the FP8 cache it quantises itself (no append): every used
    block is quantised with its valid length, then decoded from codes."""
    ids, kk, vv = snap
    local = {bid: i for i, bid in enumerate(ids)}
    bs = case.w.block_size
    maxb = max(len(t) for t in case.tables)
    tab = -np.ones((case.w.num_seqs, maxb), dtype=np.int64)
    valid = {}
    for b in seqs:
        tab[b, :len(case.tables[b])] = [local[x] for x in case.tables[b]]
        n = case.w.seq_lens[b]
        for j, x in enumerate(case.tables[b]):
            valid[local[x]] = max(valid.get(local[x], 0), min(bs, n - j * bs))
    blocks = sorted(valid)
    vl = [valid[x] for x in blocks]
    kq, ks = OQ.quantize_blocks(kk, blocks, vl)
    vq, vs = OQ.quantize_blocks(vv, blocks, vl)
    lens = np.array(case.w.seq_lens)
    return OPA.decode(_to_np64(case.q), kq, vq, tab, lens, case.w.scale,
                      k_scale=ks, v_scale=vs, seqs=list(seqs), heads=heads), (blocks, vl, ids)


def assert_close(out: torch.Tensor, ref: np.ndarray, tol: float, what=""):
    got = out.detach().to("cpu").to(torch.float64).numpy()
    m = ~np.isnan(ref)
    diff = np.abs(got[m] - ref[m])
    lim = tol + tol * np.abs(ref[m])
    bad = diff > lim
    assert not np.any(np.isnan(got[m])), f"{what}: NaN in output"
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements outside "
                           f"atol=rtol={tol}; max |diff| {diff.max():.3e}")
    return float(diff.max()) if diff.size else 0.0
