"""GPU parity of pa_decode_cascade (shared-prefix decode: the prefix's
attention computed once for every sequence's queries, each suffix by the
paged decode, merged by log-sum-exp) against the fp64 oracle, which knows
nothing of prefixes: it attends over each sequence's whole gathered cache.

Cases: the shared-prefix workload (256 forks of a 2048-token prompt) at
block sizes 8, 16 and 32 with automatic and fixed partition counts;
head_dim 64; GQA groups of 8, 1 and 3; negative and zero scales; a cascade prefix shorter than the
shared one (down to a partial last chunk); sequences that
end exactly at the prefix (prefix partial alone) and one shorter than it
(zeros, flagged); agreement with pa_decode on the same inputs.
"""
import pytest
import torch

from paged_kv_cache_228_gb300 import pa
from paged_kv_cache_228_gb300 import workloads as W

from cases import assert_close, build_case, oracle_decode, snapshot_blocks

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_228_gb300 import build
    build.build()
    pa.pa_get_device_error()


def _ws(w, splits, prefix_len):
    n = pa.pa_decode_cascade_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                            w.head_dim, w.block_size, prefix_len, splits)
    return torch.full((n,), 255, dtype=torch.uint8, device="cuda")


def _out(w):
    return torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"),
                      dtype=torch.bfloat16, device="cuda")


def _cascade(case, prefix_len, splits=0, lens=None, scale=None):
    w = case.w
    out = _out(w)
    pa.pa_decode_cascade(case.q, case.k_cache, case.v_cache, case.table_t,
                         case.lens_t if lens is None else lens, prefix_len,
                         w.scale if scale is None else scale, out,
                         _ws(w, splits, prefix_len), num_splits=splits)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("bs,splits", [(8, 0), (16, 0), (32, 0), (16, 7), (16, 2000)])
def test_cascade_parity_shared_prefix(bs, splits):
    case = build_case(W.shared_prefix(bs))
    seqs = list(range(0, case.w.num_seqs, 17)) + [case.w.num_seqs - 1]
    snap = snapshot_blocks(case, seqs)
    pa.pa_cache_write(case.k_new, case.v_new, case.slots_t, case.k_cache, case.v_cache)
    out = _cascade(case, case.w.shared_prefix, splits)
    assert_close(out, oracle_decode(case, snap, seqs), TOL, f"cascade bs{bs} splits{splits}")
    assert pa.pa_get_device_error() == 0


def test_cascade_agrees_with_decode_and_shorter_prefix():
    case = build_case(W.shared_prefix(16, num_seqs=48, prefix=512))
    w = case.w
    seqs = list(range(w.num_seqs))
    snap = snapshot_blocks(case, seqs)
    pa.pa_cache_write(case.k_new, case.v_new, case.slots_t, case.k_cache, case.v_cache)
    ref = oracle_decode(case, snap, seqs)
    dec = _out(w)
    ws = torch.empty(max(16, pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads,
                                                          w.num_kv_heads, w.head_dim)),
                     dtype=torch.uint8, device="cuda")
    pa.pa_decode(case.q, case.k_cache, case.v_cache, case.table_t, case.lens_t, w.scale, dec, ws)
    torch.cuda.synchronize()
    assert_close(dec, ref, TOL, "plain decode of the forked batch")
    for prefix_len in (512, 256, 16):   # any whole-block part of the shared prefix
        assert_close(_cascade(case, prefix_len), ref, TOL, f"cascade prefix {prefix_len}")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("sign", [-1.0, 0.0])
def test_cascade_negative_and_zero_scale(sign):
    # the prefix pass applies a negative scale as its magnitude to the
    # negated query; a zero scale weighs every token alike (also in the
    # prefix's last, partial chunk: 528 = 8 chunks + 16 tokens)
    case = build_case(W.shared_prefix(16, num_seqs=48, prefix=528))
    w = case.w
    seqs = list(range(w.num_seqs))
    snap = snapshot_blocks(case, seqs)
    pa.pa_cache_write(case.k_new, case.v_new, case.slots_t, case.k_cache, case.v_cache)
    scale = sign * w.scale
    ref = oracle_decode(case, snap, seqs, scale=scale)
    assert_close(_cascade(case, 528, scale=scale), ref, TOL, f"cascade scale {scale}")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("hq,hkv", [(8, 1), (8, 8), (12, 4)])
def test_cascade_group_sizes(hq, hkv):
    # GQA groups of 8, 1 (MHA) and 3 (not a power of two) in the prefix
    # pass's row blocks of 256 (query rows (sequence, head) of one KV head);
    # 37 sequences leave a partial last block at every group size, and a
    # 272-token prefix a partial last chunk
    base = W.shared_prefix(16, num_seqs=37, prefix=272)
    w = W.Workload(f"cascade_g{hq // hkv}", 37, hq, hkv, 128, 16, seq_lens=base.seq_lens,
                   pool_blocks=base.pool_blocks, seed=11, shared_prefix=272)
    case = build_case(w)
    seqs = list(range(w.num_seqs))
    snap = snapshot_blocks(case, seqs)
    pa.pa_cache_write(case.k_new, case.v_new, case.slots_t, case.k_cache, case.v_cache)
    ref = oracle_decode(case, snap, seqs)
    assert_close(_cascade(case, 272), ref, TOL, f"cascade G={hq // hkv}")
    assert pa.pa_get_device_error() == 0


def test_cascade_head_dim_64_and_sequences_at_the_prefix():
    # a tiny-shaped batch (d = 64, GQA 2) forked from a 64-token prompt;
    # lengths cut back so some sequences end exactly at the prefix
    base = W.shared_prefix(16, num_seqs=12, prefix=64)
    w = W.Workload("cascade_d64", 12, 4, 2, 64, 16, seq_lens=base.seq_lens,
                   pool_blocks=base.pool_blocks, seed=9, shared_prefix=64)
    case = build_case(w)
    seqs = list(range(w.num_seqs))
    snap = snapshot_blocks(case, seqs)  # before any library kernel writes the pool
    pa.pa_cache_write(case.k_new, case.v_new, case.slots_t, case.k_cache, case.v_cache)
    lens = list(w.seq_lens)
    lens[0] = lens[5] = 64
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = _cascade(case, 64, lens=lens_t)
    # the oracle applies the append to the snapshot and attends over `lens`
    ref = oracle_decode(case, snap, seqs, lens=lens)
    assert_close(out, ref, TOL, "cascade d64 with sequences at the prefix")
    assert pa.pa_get_device_error() == 0
    # a sequence shorter than the prefix: zeros and a flag
    lens[3] = 48
    out = _cascade(case, 64, lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    assert pa.pa_get_device_error() & pa.DEVERR_BAD_SEQ_LEN
    assert torch.all(out[3] == 0)


@pytest.mark.parametrize("bs", [64, 256])
def test_cascade_large_blocks(bs):
    # blocks larger than a prefix chunk (256: two chunks per block, read at
    # an offset inside it) and at half a chunk (64)
    case = build_case(W.shared_prefix(bs, num_seqs=40, prefix=512))
    w = case.w
    seqs = list(range(w.num_seqs))
    snap = snapshot_blocks(case, seqs)
    pa.pa_cache_write(case.k_new, case.v_new, case.slots_t, case.k_cache, case.v_cache)
    ref = oracle_decode(case, snap, seqs)
    for prefix_len in (512, 256):
        if prefix_len % bs == 0:
            assert_close(_cascade(case, prefix_len), ref, TOL, f"cascade bs{bs} prefix {prefix_len}")
    assert pa.pa_get_device_error() == 0
