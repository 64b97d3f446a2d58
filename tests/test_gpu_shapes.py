"""GPU parity of pa_decode on shapes the named workloads do not cover, all
against the fp64 oracle (bf16 1e-2, FP8 5e-2):

* MQA: 8 query heads on one KV head, 300 sequences (the length scan takes
  several 128-sequence passes), block size 32;
* MHA: group 1, block size 256 (the largest), d = 64;
* a group of 3 (not a power of two), block size 8;
* one 256K-token sequence on one KV head, split across every CTA (sampled
  heads checked), bf16 and FP8;
* 2048 sequences of 1..70 tokens (dozens of whole segments per CTA, query
  slots reused many times, 16 passes of the length scan), bf16 and FP8.
"""
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_228_gb300 import pa
from paged_kv_cache_228_gb300 import workloads as W

from cases import assert_close, build_case, oracle_decode, oracle_decode_fp8, snapshot_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_228_gb300 import build
    build.build()
    pa.pa_get_device_error()


def _workload(name, B, hq, hkv, d, bs, lens, seed):
    need = sum(-(-n // bs) for n in lens)
    return W.Workload(name, B, hq, hkv, d, bs, seq_lens=lens,
                      pool_blocks=math.ceil(1.3 * need) + 2, seed=seed)


def _run(case, splits=0, **kw):
    w = case.w
    pa.pa_cache_write(case.k_new, case.v_new, case.slots_t, case.k_cache, case.v_cache)
    out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    n = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                    splits)
    ws = torch.full((max(16, n),), 255, dtype=torch.uint8, device="cuda")
    pa.pa_decode(case.q, case.k_cache, case.v_cache, case.table_t, case.lens_t, w.scale, out,
                 ws, num_splits=splits, **kw)
    torch.cuda.synchronize()
    return out


def _lens(B, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


@pytest.mark.parametrize("name,B,hq,hkv,d,bs,lo,hi", [
    ("mqa", 300, 8, 1, 128, 32, 1, 600),
    ("mha_bs256", 5, 4, 4, 64, 256, 200, 1500),
    ("gqa3_bs8", 40, 6, 2, 128, 8, 1, 700),
])
def test_shape_parity(name, B, hq, hkv, d, bs, lo, hi):
    w = _workload(name, B, hq, hkv, d, bs, _lens(B, lo, hi, 7), 21)
    case = build_case(w, poison_unused=True)
    seqs = range(B)
    snap = snapshot_blocks(case, seqs)
    for splits in (0, 3):
        out = _run(case, splits) if splits == 0 else _rerun(case, splits)
        assert_close(out, oracle_decode(case, snap, seqs), 1e-2, f"{name} splits {splits}")
    assert pa.pa_get_device_error() == 0


def _rerun(case, splits):
    # the cache already holds the appended token: decode only
    w = case.w
    out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    n = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                    splits)
    ws = torch.full((max(16, n),), 255, dtype=torch.uint8, device="cuda")
    pa.pa_decode(case.q, case.k_cache, case.v_cache, case.table_t, case.lens_t, w.scale, out,
                 ws, num_splits=splits)
    torch.cuda.synchronize()
    return out


def test_one_256k_sequence_bf16_and_fp8():
    n = 262144
    w = _workload("long1", 1, 8, 1, 64, 16, [n], 23)
    case = build_case(w)
    snap = snapshot_blocks(case, [0])
    out = _run(case)
    assert_close(out, oracle_decode(case, snap, [0]), 1e-2, "256K bf16")
    assert pa.pa_get_device_error() == 0
    # FP8: the oracle quantises the blocks itself (valid lengths from the
    # post-append cache), the GPU quantises the same blocks
    ref, (blocks, vl, ids) = oracle_decode_fp8(case, snapshot_blocks(case, [0]), [0])
    phys = torch.tensor([ids[b] for b in blocks], dtype=torch.int32, device="cuda")
    kq = torch.zeros(case.k_cache.shape, dtype=torch.uint8, device="cuda")
    vq = torch.zeros_like(kq)
    ks = torch.ones((w.pool_blocks, 1), device="cuda")
    vs = torch.ones_like(ks)
    pa.pa_quantize_fp8(case.k_cache, case.v_cache, phys,
                       torch.tensor(vl, dtype=torch.int32, device="cuda"), kq, vq, ks, vs)
    out8 = torch.full_like(out, float("nan"))
    nws = pa.pa_decode_workspace_size(1, 8, 1, 64)
    ws = torch.full((max(16, nws),), 255, dtype=torch.uint8, device="cuda")
    pa.pa_decode(case.q, kq, vq, case.table_t, case.lens_t, w.scale, out8, ws,
                 k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert_close(out8, ref, 5e-2, "256K fp8")
    assert pa.pa_get_device_error() == 0


def test_many_short_sequences_bf16_fp8():
    # 2048 sequences of 1..70 tokens: every CTA walks dozens of whole
    # segments (query-slot reuse, segment hand-over in the copy warp), and
    # the length scan takes 16 passes of 128.
    B = 2048
    w = _workload("short", B, 16, 4, 128, 16, _lens(B, 1, 70, 11), 25)
    case = build_case(w, poison_unused=True)
    seqs = list(range(0, B, 41))
    snap = snapshot_blocks(case, seqs)
    out = _run(case)
    assert_close(out, oracle_decode(case, snap, seqs), 1e-2, "short bf16")
    assert pa.pa_get_device_error() == 0
    ref, (blocks, vl, ids) = oracle_decode_fp8(case, snapshot_blocks(case, seqs), seqs)
    phys = torch.tensor([ids[b] for b in blocks], dtype=torch.int32, device="cuda")
    kq = torch.zeros(case.k_cache.shape, dtype=torch.uint8, device="cuda")
    vq = torch.zeros_like(kq)
    ks = torch.ones((w.pool_blocks, w.num_kv_heads), device="cuda")
    vs = torch.ones_like(ks)
    pa.pa_quantize_fp8(case.k_cache, case.v_cache, phys,
                       torch.tensor(vl, dtype=torch.int32, device="cuda"), kq, vq, ks, vs)
    out8 = torch.full_like(out, float("nan"))
    nws = pa.pa_decode_workspace_size(B, 16, 4, 128)
    ws = torch.full((max(16, nws),), 255, dtype=torch.uint8, device="cuda")
    pa.pa_decode(case.q, kq, vq, case.table_t, case.lens_t, w.scale, out8, ws,
                 k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert_close(out8, ref, 5e-2, "short fp8")
    assert pa.pa_get_device_error() == 0
