"""The FP8 decode's query split, measured on its own.

The E4M3 tensor-core paths take the query as two E4M3 terms per head: with
the power of two 2^s that puts max|q_h| * 2^s in [128, 256),
    x = q * 2^s,   hi = e4m3(x),   lo = e4m3(16 (x - hi)),
and the scores use (hi + lo / 16) / 2^s.  Here the split is written from
that definition, with the oracle's E4M3 codec for the code arithmetic.

* For a bf16 query the split is exact wherever |x| >= 2^-6 (elements above
  about 2^-14 of the row's largest): a bf16 value has 8 significant bits;
  rounding to E4M3's 4 leaves a residual of at most 4 bits on a grid E4M3
  still reaches.  Below that the lo term is subnormal and the error is at
  most 2^-14 in units of x.  So the query costs the decode nothing
  measurable: the oracle's decode with the split query equals the exact
  query's to 1e-9 on the tiny workload.
* For fp32 values (the softmax weights P' take the same split) the bound is
  |hi + lo / 16 - x| <= 2^-8 |x| + 2^-14.
"""
import numpy as np
import torch

from oracle import e4m3 as E
from oracle import paged_attention as OPA
from oracle import quantize as OQ
from paged_kv_cache_228_gb300 import workloads as W

from cases import _to_np64, build_case, snapshot_blocks


def split_rows(q):
    """(q', x, hi, lo): the two-term E4M3 split of each row of q (float64,
    last axis = head dim) and its value q' = (hi + lo / 16) / 2^s."""
    amax = np.abs(q).max(axis=-1, keepdims=True)
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) + 1, -100)
    qs = 2.0 ** (8 - e)  # max |x| in [128, 256)
    x = q * qs
    hi = E.decode(E.encode_fast(x))
    lo = E.decode(E.encode_fast(16.0 * (x - hi)))
    return (hi + lo / 16.0) / qs, x, hi, lo


def _rows(rng, n, d, spread):
    return rng.standard_normal((n, d)) * np.exp2(rng.integers(-spread, spread, (n, 1))) * \
        np.exp2(rng.uniform(-20, 0, (n, d)))


def test_bf16_query_split_is_exact_above_the_subnormal_floor():
    rng = np.random.default_rng(7)
    q = torch.tensor(_rows(rng, 256, 128, 12)).to(torch.bfloat16).double().numpy()
    _, x, hi, lo = split_rows(q)
    amax = np.abs(x).max(axis=-1)
    assert np.all((amax >= 128) & (amax < 256))
    err = np.abs(hi + lo / 16.0 - x)
    big = np.abs(x) >= 2.0 ** -6
    assert big.sum() > 0.5 * big.size and (~big).sum() > 0  # both regimes occur
    assert np.all(err[big] == 0.0)
    assert np.all(err[~big] <= 2.0 ** -14)


def test_fp32_split_bound():
    rng = np.random.default_rng(8)
    p = _rows(rng, 256, 128, 12).astype(np.float32).astype(np.float64)
    _, x, hi, lo = split_rows(p)
    err = np.abs(hi + lo / 16.0 - x)
    bound = 2.0 ** -8 * np.abs(x) + 2.0 ** -14
    assert np.all(err <= bound)
    assert np.max(err / bound) > 0.25  # the bound is not loose


def test_query_split_costs_the_decode_nothing():
    case = build_case(W.tiny(), device="cpu")
    seqs = list(range(case.w.num_seqs))
    ids, kk, vv = snapshot_blocks(case, seqs)
    local = {bid: i for i, bid in enumerate(ids)}
    bs = case.w.block_size
    tab = -np.ones((case.w.num_seqs, max(len(t) for t in case.tables)), dtype=np.int64)
    valid = {}
    for b in seqs:
        tab[b, :len(case.tables[b])] = [local[x] for x in case.tables[b]]
        for j, x in enumerate(case.tables[b]):
            valid[local[x]] = max(valid.get(local[x], 0), min(bs, case.w.seq_lens[b] - j * bs))
    blocks = sorted(valid)
    kq, ks = OQ.quantize_blocks(kk, blocks, [valid[x] for x in blocks])
    vq, vs = OQ.quantize_blocks(vv, blocks, [valid[x] for x in blocks])
    lens = np.array(case.w.seq_lens)
    q = _to_np64(case.q)
    kw = dict(k_scale=ks, v_scale=vs, seqs=seqs)
    ref = OPA.decode(q, kq, vq, tab, lens, case.w.scale, **kw)
    ref_split = OPA.decode(split_rows(q)[0], kq, vq, tab, lens, case.w.scale, **kw)
    d = np.nanmax(np.abs(ref_split - ref))
    print(f"tiny FP8: max |decode(split q) - decode(q)| = {d:.2e}")
    assert d <= 1e-9
