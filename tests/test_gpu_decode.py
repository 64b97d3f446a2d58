"""GPU parity of pa_decode (after the step's pa_cache_write) against the
fp64 oracle, through the C ABI, plus invariants that pin the kernel's
gather and split logic:

* every workload shape: tiny (B=4, GQA 2, d=64, 32-block pool), the
  Llama-3.2-1B and Llama-3.1-8B shaped layers in full, the shared-prefix
  shape at block sizes 8, 16, 32 (sampled sequences), and the 70B / 128K
  long-context layer (sampled sequences and heads, bf16 and FP8);
* tolerance: |out - ref| <= 1e-2 + 1e-2 |ref| for bf16 caches and 5e-2 for
  FP8 caches against the oracle run on the cache it quantises itself;
* seq_len = 1 returns the V row exactly; permuting physical block ids and
  replacing shared prefix blocks by copies give bit-identical outputs; the
  work-partition count changes nothing beyond tolerance; empty sequences
  give zeros; NaN-poisoned unused slots and blocks are never read; bad
  table entries and lengths are flagged on the device error word.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_228_gb300 import pa
from paged_kv_cache_228_gb300 import workloads as W

from cases import assert_close, build_case, oracle_decode, oracle_decode_fp8, snapshot_blocks

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2
TOL_FP8 = 5e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_228_gb300 import build
    build.build()
    pa.pa_get_device_error()


def _workspace(case, num_splits=0):
    w = case.w
    n = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                    num_splits)
    # 0xFF bytes read as NaN: a partial the kernels never wrote would show up
    return torch.full((max(n, 16),), 255, dtype=torch.uint8, device="cuda")


def run_step(case, num_splits=0, write=True, k_cache=None, v_cache=None, k_scale=None,
             v_scale=None, table=None):
    """pa_cache_write of the append step, then pa_decode; returns out."""
    w = case.w
    kc = case.k_cache if k_cache is None else k_cache
    vc = case.v_cache if v_cache is None else v_cache
    if write:
        pa.pa_cache_write(case.k_new, case.v_new, case.slots_t, kc, vc)
    out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    pa.pa_decode(case.q, kc, vc, case.table_t if table is None else table, case.lens_t,
                 w.scale, out, _workspace(case, num_splits), k_scale=k_scale,
                 v_scale=v_scale, num_splits=num_splits)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name", ["tiny", "llama3.2-1b", "llama3.1-8b"])
def test_decode_parity_full(name):
    case = build_case(W.WORKLOADS[name](), poison_unused=True)
    seqs = range(case.w.num_seqs)
    snap = snapshot_blocks(case, seqs)
    out = run_step(case)
    ref = oracle_decode(case, snap, seqs)
    assert_close(out, ref, TOL_BF16, name)
    assert pa.pa_get_device_error() == 0


def test_tiny_decode_before_and_after_append():
    # decode at lengths {7, 16, 33, 50}, append one token each, decode again
    w = W.tiny()
    case = build_case(w)
    seqs = range(4)
    snap = snapshot_blocks(case, seqs)
    pre = W.Workload(**{**w.__dict__, "seq_lens": [n - 1 for n in w.seq_lens]})
    pre_case = build_case(w)
    pre_case.w = pre
    pre_case.lens_t = torch.tensor(pre.seq_lens, dtype=torch.int32, device="cuda")
    out0 = run_step(pre_case, write=False)
    ref0 = oracle_decode(pre_case, snap, seqs, with_append=False)
    assert_close(out0, ref0, TOL_BF16, "tiny pre-append")
    out1 = run_step(case)
    ref1 = oracle_decode(case, snap, seqs)
    assert_close(out1, ref1, TOL_BF16, "tiny post-append")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_decode_parity_shared_prefix(bs):
    case = build_case(W.shared_prefix(bs))
    seqs = [0, 1, 77, 128, 255]
    snap = snapshot_blocks(case, seqs)
    out = run_step(case)
    ref = oracle_decode(case, snap, seqs)
    assert_close(out, ref, TOL_BF16, f"shared prefix bs={bs}")
    assert pa.pa_get_device_error() == 0


@pytest.fixture(scope="module")
def long_case():
    return build_case(W.llama31_70b_128k())


def test_decode_parity_70b_128k_bf16(long_case):
    case = long_case
    seqs = [5]
    heads = list(range(0, 64, 7))
    snap = snapshot_blocks(case, seqs)
    out = run_step(case)
    ref = oracle_decode(case, snap, seqs, heads=heads)
    assert_close(out, ref, TOL_BF16, "70b 128k bf16")
    assert pa.pa_get_device_error() == 0


def test_decode_parity_70b_128k_fp8(long_case):
    case = long_case
    w = case.w
    seqs = [3]
    heads = [0, 9, 18, 27, 36, 45, 54, 63]
    snap = snapshot_blocks(case, seqs)
    # quantise every block of the pool (full blocks: 131072 = 8192 * 16)
    kq = torch.empty(case.k_cache.shape, dtype=torch.uint8, device="cuda")
    vq = torch.empty_like(kq)
    ks = torch.empty((w.pool_blocks, w.num_kv_heads), device="cuda")
    vs = torch.empty_like(ks)
    ids = torch.arange(w.pool_blocks, dtype=torch.int32, device="cuda")
    valid = torch.full((w.pool_blocks,), w.block_size, dtype=torch.int32, device="cuda")
    pa.pa_quantize_fp8(case.k_cache, case.v_cache, ids, valid, kq, vq, ks, vs)
    out = run_step(case, write=False, k_cache=kq, v_cache=vq, k_scale=ks, v_scale=vs)
    ref, _ = oracle_decode_fp8(case, snap, seqs, heads=heads)
    assert_close(out, ref, TOL_FP8, "70b 128k fp8")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("name,bs", [("llama3.1-8b", 16), ("shared_prefix", 8),
                                     ("shared_prefix", 32), ("shared_prefix", 64),
                                     ("llama3.2-1b", 16)])
def test_decode_parity_fp8(name, bs):
    w = W.shared_prefix(bs) if name == "shared_prefix" else W.WORKLOADS[name]()
    case = build_case(w)
    seqs = list(range(0, w.num_seqs, max(1, w.num_seqs // 12)))
    snap = snapshot_blocks(case, seqs)
    ref, (blocks, vl, ids) = oracle_decode_fp8(case, snap, seqs)
    # quantise on the GPU the same blocks with the same valid lengths
    phys = torch.tensor([ids[b] for b in blocks], dtype=torch.int32, device="cuda")
    kq = torch.zeros(case.k_cache.shape, dtype=torch.uint8, device="cuda")
    vq = torch.zeros_like(kq)
    ks = torch.ones((w.pool_blocks, w.num_kv_heads), device="cuda")
    vs = torch.ones_like(ks)
    pa.pa_quantize_fp8(case.k_cache, case.v_cache, phys,
                       torch.tensor(vl, dtype=torch.int32, device="cuda"), kq, vq, ks, vs)
    out = run_step(case, write=False, k_cache=kq, v_cache=vq, k_scale=ks, v_scale=vs)
    assert_close(out, ref, TOL_FP8, f"{name} fp8")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("bs", [16, 8])
def test_decode_parity_fp8_large_v_scales(bs):
    # Every other block's V is scaled by 300 (V scales up to ~0.7): FP8
    # tiles whose V scale is >= 0.5 take the normalised-P path, the rest
    # put the scale into P; both mix within a sequence (and, at bs 8,
    # within a tile).
    w = W.shared_prefix(bs, num_seqs=24, prefix=256) if bs == 8 else W.llama32_1b(24)
    case = build_case(w)
    case.v_cache[::2] = (case.v_cache[::2].float() * 300.0).to(torch.bfloat16)
    seqs = list(range(w.num_seqs))
    snap = snapshot_blocks(case, seqs)
    ref, (blocks, vl, ids) = oracle_decode_fp8(case, snap, seqs)
    phys = torch.tensor([ids[b] for b in blocks], dtype=torch.int32, device="cuda")
    kq = torch.zeros(case.k_cache.shape, dtype=torch.uint8, device="cuda")
    vq = torch.zeros_like(kq)
    ks = torch.ones((w.pool_blocks, w.num_kv_heads), device="cuda")
    vs = torch.ones_like(ks)
    pa.pa_quantize_fp8(case.k_cache, case.v_cache, phys,
                       torch.tensor(vl, dtype=torch.int32, device="cuda"), kq, vq, ks, vs)
    assert float(vs.max()) >= 0.5 and float(vs[phys.long()].min()) < 0.5
    out = run_step(case, write=False, k_cache=kq, v_cache=vq, k_scale=ks, v_scale=vs)
    assert_close(out, ref, TOL_FP8, f"fp8 large V scales bs{bs}")
    assert pa.pa_get_device_error() == 0


def test_seq_len_one_returns_v_exactly():
    w = W.Workload("one", 6, 16, 4, 128, 16, seq_lens=[1] * 6, pool_blocks=64, seed=9)
    case = build_case(w)
    out = run_step(case)
    v = case.v_cache.float()
    for b in range(6):
        blk = case.tables[b][0]
        for h in range(16):
            assert torch.equal(out[b, h].float(), v[blk, h // 4, 0]), (b, h)


def _permuted(case, seed):
    """Same logical contents under a random relabelling of physical blocks."""
    nb = case.w.pool_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(seed))
    kc = torch.empty_like(case.k_cache)
    vc = torch.empty_like(case.v_cache)
    kc[perm.cuda()] = case.k_cache
    vc[perm.cuda()] = case.v_cache
    tab = case.table_t.clone().long()
    m = tab >= 0
    tab[m] = perm.cuda()[tab[m]]
    return kc, vc, tab.int()


@pytest.mark.parametrize("name", ["llama3.1-8b", "shared_prefix_bs8"])
def test_physical_permutation_is_bit_identical(name):
    case = build_case(W.WORKLOADS[name]())
    out = run_step(case, write=False)
    kc, vc, tab = _permuted(case, 5)
    out2 = run_step(case, write=False, k_cache=kc, v_cache=vc, table=tab)
    assert torch.equal(out, out2)


def test_shared_vs_copied_prefix_is_bit_identical():
    w = W.shared_prefix(16, num_seqs=16)
    w.pool_blocks = 16 * (2048 // 16) + 16 * 33 + 64   # room for private copies
    case = build_case(w)
    out = run_step(case, write=False)
    # give every sequence private copies of the prefix blocks
    npre = w.shared_prefix // w.block_size
    free = sorted(set(range(w.pool_blocks)) - {b for t in case.tables for b in t})
    assert len(free) >= npre * (w.num_seqs - 1)
    tab = case.table_t.clone()
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    i = 0
    for b in range(1, w.num_seqs):
        for j in range(npre):
            nbk = free[i]
            i += 1
            src = case.tables[b][j]
            kc[nbk] = kc[src]
            vc[nbk] = vc[src]
            tab[b, j] = nbk
    out2 = run_step(case, write=False, k_cache=kc, v_cache=vc, table=tab)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("splits", [1, 2, 7, 151, 2000])
def test_partition_count_within_tolerance(splits):
    case = build_case(W.llama31_8b())
    seqs = range(0, 128, 9)
    snap = snapshot_blocks(case, seqs)
    out = run_step(case, num_splits=splits)
    ref = oracle_decode(case, snap, seqs)
    assert_close(out, ref, TOL_BF16, f"splits={splits}")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("splits", [0, 2000])
def test_repeated_decode_is_bit_identical(splits):
    # The reduction order depends only on logical positions and the partition
    # count, so repeated calls must agree bit for bit; a pipeline race (a tile
    # read before its copy landed or after the next copy overwrote it) would
    # show up here as run-to-run differences.
    case = build_case(W.llama31_8b())
    outs = [run_step(case, write=False, num_splits=splits) for _ in range(6)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert pa.pa_get_device_error() == 0


def test_empty_and_ragged_sequences():
    lens = [0, 1, 15, 16, 17, 0, 33, 255, 256, 257]
    w = W.Workload("ragged", len(lens), 8, 2, 64, 16, seq_lens=[max(1, n) for n in lens],
                   pool_blocks=64, seed=21)
    case = build_case(w)
    case.w.seq_lens = lens
    case.lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    seqs = range(len(lens))
    snap = snapshot_blocks(case, seqs)
    out = run_step(case, write=False)
    ref = oracle_decode(case, snap, seqs, with_append=False)
    assert_close(out, ref, TOL_BF16, "ragged")
    assert torch.equal(out[0], torch.zeros_like(out[0]))
    assert pa.pa_get_device_error() == 0


def test_bad_table_entry_and_length_are_flagged():
    case = build_case(W.tiny())
    tab = case.table_t.clone()
    tab[2, 1] = 10 ** 6
    out = run_step(case, write=False, table=tab)
    assert pa.pa_get_device_error() & pa.DEVERR_BAD_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    lens = case.lens_t.clone()
    case.lens_t = torch.tensor([8, 17, 34, 10 ** 6], dtype=torch.int32, device="cuda")
    run_step(case, write=False)
    assert pa.pa_get_device_error() & pa.DEVERR_BAD_SEQ_LEN
    case.lens_t = lens
    assert pa.pa_get_device_error() == 0


def test_workspace_too_small_is_rejected():
    case = build_case(W.tiny())
    w = case.w
    out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.bfloat16,
                      device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode(case.q, case.k_cache, case.v_cache, case.table_t, case.lens_t, w.scale,
                     out, torch.empty(16, dtype=torch.uint8, device="cuda"), num_splits=4)
    assert e.value.status == pa.PA_ERR_WORKSPACE


@pytest.mark.parametrize("splits", [1, 5, 37, 2000])
def test_more_partitions_than_tiles(splits):
    # The tiny batch has 2 * (1 + 2 + 3 + 4) = 20 tiles: with more partitions
    # than tiles only the first W CTAs take part, one tile each, and nearly
    # every segment goes through the merge.
    case = build_case(W.tiny(), poison_unused=True)
    seqs = range(case.w.num_seqs)
    snap = snapshot_blocks(case, seqs)
    out = run_step(case, num_splits=splits)
    assert_close(out, oracle_decode(case, snap, seqs), TOL_BF16, f"tiny splits={splits}")
    assert pa.pa_get_device_error() == 0


# ------------------------------------------------ FP8, head_dim 128 paths ---
def _fp8_cache(case, seqs, poison=False):
    """The oracle's FP8 reference for `seqs` and a GPU E4M3 cache of the same
    blocks quantised by the library; with poison, every code past a block's
    valid tokens is an E4M3 NaN (0x7F), which the kernel must never let into
    a product."""
    w = case.w
    snap = snapshot_blocks(case, seqs)
    ref, (blocks, vl, ids) = oracle_decode_fp8(case, snap, seqs)
    phys = torch.tensor([ids[b] for b in blocks], dtype=torch.int32, device="cuda")
    kq = torch.zeros(case.k_cache.shape, dtype=torch.uint8, device="cuda")
    vq = torch.zeros_like(kq)
    ks = torch.ones((w.pool_blocks, w.num_kv_heads), device="cuda")
    vs = torch.ones_like(ks)
    pa.pa_quantize_fp8(case.k_cache, case.v_cache, phys,
                       torch.tensor(vl, dtype=torch.int32, device="cuda"), kq, vq, ks, vs)
    if poison:
        for b, n in zip(phys.tolist(), vl):
            kq[b, :, n:, :] = 0x7F
            vq[b, :, n:, :] = 0x7F
    return ref, kq, vq, ks, vs


@pytest.mark.parametrize("splits", [1, 7, 151, 2000])
def test_fp8_partition_count_within_tolerance(splits):
    case = build_case(W.llama31_8b())
    ref, kq, vq, ks, vs = _fp8_cache(case, list(range(0, 128, 9)))
    out = run_step(case, num_splits=splits, write=False, k_cache=kq, v_cache=vq, k_scale=ks,
                   v_scale=vs)
    assert_close(out, ref, TOL_FP8, f"fp8 splits={splits}")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("splits", [0, 2000])
def test_fp8_repeated_decode_is_bit_identical(splits):
    case = build_case(W.llama31_8b())
    _, kq, vq, ks, vs = _fp8_cache(case, list(range(0, 128, 9)))
    outs = [run_step(case, write=False, num_splits=splits, k_cache=kq, v_cache=vq, k_scale=ks,
                     v_scale=vs) for _ in range(6)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_fp8_empty_and_ragged_sequences_poisoned_tails(bs):
    # lengths around the 16-token tile, the 32-token MMA step, the 128-token
    # half chunk and the 256-token chunk (the tensor-core kernel's work
    # unit); the codes past each sequence's end are NaN
    lens = [0, 1, 15, 16, 17, 31, 32, 33, 127, 128, 129, 0, 255, 256, 257, 300, 511, 512,
            513, 767, 768, 769]
    w = W.Workload("ragged128", len(lens), 32, 8, 128, bs,
                   seq_lens=[max(1, n) for n in lens],
                   pool_blocks=sum(-(-max(1, n) // bs) for n in lens) + 8, seed=22)
    case = build_case(w)
    case.w.seq_lens = lens
    case.lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    seqs = [b for b, n in enumerate(lens) if n > 0]
    ref, kq, vq, ks, vs = _fp8_cache(case, seqs, poison=True)
    out = run_step(case, write=False, k_cache=kq, v_cache=vq, k_scale=ks, v_scale=vs)
    assert_close(out, ref, TOL_FP8, f"fp8 ragged bs{bs}")
    assert torch.equal(out[0], torch.zeros_like(out[0]))
    assert torch.equal(out[11], torch.zeros_like(out[11]))
    assert pa.pa_get_device_error() == 0
