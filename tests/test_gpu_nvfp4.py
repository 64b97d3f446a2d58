"""GPU parity of the NVFP4 cache path (pa_cache_write_nvfp4, pa_decode_nvfp4)
against the oracle's NVFP4 restatement, through the C ABI.

* cache write: every byte of the four pools (values, block scales, for K and
  V) equals the oracle's, for head_dim 64 and 128, block sizes 16 and 32, the
  workload shapes, rows with zeros, values that round to E4M3 zero scales,
  saturating rows, exact E2M1 midpoints and signed zeros, and slots written
  out of order with skipped (-1) tokens;
* decode: |out - ref| <= 1e-2 + 1e-2 |ref| against the fp64 oracle decoding
  the oracle's own quantised cache (the kernel's K and V values are exact in
  f16; q is rounded to f16, P to f16, the output to bf16), full outputs for
  the small shapes and sampled sequences / heads for the large ones
  including the 70B / 128K layer; unused slots and blocks hold NaN block
  scales and must never reach the output;
* empty and ragged sequences, every work-partition count within tolerance and
  repeated calls bit-identical, out-of-pool table entries and slots flagged;
* shapes beyond the workloads: MQA over 300 sequences, MHA at block size 256,
  a group of 3, one 256K-token sequence split across every CTA, and 2048
  sequences of 1..70 tokens;
* the fused append (pa_decode_append_nvfp4) equals write then decode bit for
  bit, and skips or flags slots as pa_decode_append does.
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4 as ON
from paged_kv_cache_228_gb300 import pa
from paged_kv_cache_228_gb300 import workloads as W

from cases import assert_close, build_case, snapshot_blocks

pytestmark = pytest.mark.gpu

TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_228_gb300 import build
    build.build()
    pa.pa_get_device_error()


def _np(t):
    return t.detach().to("cpu").numpy()


def gscales(snap):
    """Tensor scales amax / (6 * 448) of the sampled blocks (host fp32)."""
    _, kk, vv = snap
    return (float(np.float32(np.abs(kk).max() / 2688.0)),
            float(np.float32(np.abs(vv).max() / 2688.0)))


def gpu_pool(case, k_gs, v_gs):
    """NVFP4 pools with every slot of the case's bf16 pool quantised."""
    w = case.w
    nb, bs, h, d = w.pool_blocks, w.block_size, w.num_kv_heads, w.head_dim
    cache = pa.nvfp4_empty_cache(nb, h, bs, d)
    rk = case.k_cache.permute(0, 2, 1, 3).reshape(nb * bs, h, d).contiguous()
    rv = case.v_cache.permute(0, 2, 1, 3).reshape(nb * bs, h, d).contiguous()
    slots = torch.arange(nb * bs, dtype=torch.int64, device="cuda")
    pa.pa_cache_write_nvfp4(rk, rv, slots, cache, k_gs, v_gs)
    del rk, rv
    torch.cuda.synchronize()
    return cache


def oracle_pool(snap, k_gs, v_gs):
    """The oracle's NVFP4 pools of the snapshot blocks (local ids)."""
    _, kk, vv = snap
    n, h, bs, d = kk.shape
    rk = kk.transpose(0, 2, 1, 3).reshape(n * bs, h, d)
    rv = vv.transpose(0, 2, 1, 3).reshape(n * bs, h, d)
    return ON.cache_write(rk, rv, np.arange(n * bs), ON.empty_cache(n, h, bs, d), k_gs, v_gs)


def assert_pool_equal(cache, ocache, ids):
    """GPU blocks ids[i] against the oracle's local blocks i, i < len(ids)."""
    idx = torch.tensor(ids, dtype=torch.int64, device="cuda")
    for name, g, o in zip(("k", "k_sf", "v", "v_sf"), cache, ocache):
        o = o[:len(ids)]
        got = _np(g.index_select(0, idx))
        bad = np.argwhere(got != o)
        assert bad.size == 0, f"{name}: {len(bad)} bytes differ, first at {bad[0]}"


def poison_unused(cache, case):
    """NaN block scales (E4M3 0x7F) and -6 codes in every slot no sequence
    reads: past each sequence's end in its last block, and unused blocks."""
    k, k_sf, v, v_sf = cache
    w = case.w
    used = torch.zeros(w.pool_blocks, dtype=torch.bool)
    for t in case.tables:
        used[t] = True
    un = (~used).nonzero().flatten().to("cuda")
    for a in cache:
        a[un] = 0x7F if a is k_sf or a is v_sf else 0xFF
    for b, t in enumerate(case.tables):
        tail = w.seq_lens[b] % w.block_size
        if tail:
            k_sf[t[-1], :, tail:] = 0x7F
            v_sf[t[-1], :, :, tail:] = 0x7F
            k[t[-1], :, tail:] = 0xFF


def oracle_out(case, snap, ocache, k_gs, v_gs, seqs, heads=None):
    ids = snap[0]
    local = {bid: i for i, bid in enumerate(ids)}
    maxb = max(len(t) for t in case.tables)
    tab = -np.ones((case.w.num_seqs, maxb), dtype=np.int64)
    for b in seqs:
        tab[b, :len(case.tables[b])] = [local[x] for x in case.tables[b]]
    q = case.q.to("cpu").to(torch.float64).numpy()
    return ON.decode(q, ocache, k_gs, v_gs, tab, np.array(case.w.seq_lens), case.w.scale,
                     seqs=list(seqs), heads=heads)


def run_decode(case, cache, k_gs, v_gs, num_splits=0, table=None, lens=None):
    w = case.w
    n = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                    num_splits)
    ws = torch.full((max(n, 16),), 255, dtype=torch.uint8, device="cuda")
    out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    pa.pa_decode_nvfp4(case.q, cache, k_gs, v_gs, case.table_t if table is None else table,
                       case.lens_t if lens is None else lens, w.scale, out, ws,
                       num_splits=num_splits)
    torch.cuda.synchronize()
    return out


def _seqs(w, cap=12):
    return list(range(0, w.num_seqs, max(1, w.num_seqs // cap)))


@pytest.mark.parametrize("name", ["tiny", "llama3.2-1b", "llama3.1-8b", "shared_prefix_bs32"])
def test_write_bit_exact_and_decode_parity(name):
    case = build_case(W.WORKLOADS[name]())
    w = case.w
    seqs = list(range(w.num_seqs)) if w.num_seqs <= 8 else _seqs(w)
    snap = snapshot_blocks(case, seqs)
    k_gs, v_gs = gscales(snap)
    cache = gpu_pool(case, k_gs, v_gs)
    ocache = oracle_pool(snap, k_gs, v_gs)
    assert_pool_equal(cache, ocache, snap[0])
    poison_unused(cache, case)
    out = run_decode(case, cache, k_gs, v_gs)
    ref = oracle_out(case, snap, ocache, k_gs, v_gs, seqs)
    assert_close(out, ref, TOL, f"nvfp4 {name}")
    assert pa.pa_get_device_error() == 0


def test_70b_128k_sampled():
    case = build_case(W.llama31_70b_128k())
    seqs, heads = [6], [1, 10, 19, 28, 37, 46, 55, 62]
    snap = snapshot_blocks(case, seqs)
    k_gs, v_gs = gscales(snap)
    cache = gpu_pool(case, k_gs, v_gs)
    case.k_cache = case.v_cache = None  # the bf16 pool is no longer needed
    ocache = oracle_pool(snap, k_gs, v_gs)
    # the sequence's first 64 blocks, byte for byte
    assert_pool_equal(cache, ocache, snap[0][:64])
    out = run_decode(case, cache, k_gs, v_gs)
    ref = oracle_out(case, snap, ocache, k_gs, v_gs, seqs, heads=heads)
    assert_close(out, ref, TOL, "nvfp4 70b 128k")
    assert pa.pa_get_device_error() == 0


def _special_rows(g, T, h, d):
    """Rows exercising the encoder's edge cases (see the module docstring)."""
    x = g.standard_normal((T, h, d)).astype(np.float32)
    x[0] = 0.0                                          # all-zero groups
    x[1] = 2.0 ** -30                                   # block scale rounds to 0
    x[2] = np.float32(3e4) * np.sign(x[2])              # saturating scale
    x[3, :, ::16] = 6.0                                 # exact midpoints with scale 1:
    x[3, :, 1::16] = 2.5                                # 2.5 -> 2, 5 -> 4, .25 -> 0,
    x[3, :, 2::16] = 5.0                                # 1.75 -> 2, -0.25 -> -0
    x[3, :, 3::16] = 0.25
    x[3, :, 4::16] = 1.75
    x[3, :, 5::16] = -0.25
    x[4] = -0.0                                         # negative zeros
    x[5, :, :8] = 1e-3                                  # one tiny and one normal group
    return torch.from_numpy(x).to(torch.bfloat16)


@pytest.mark.parametrize("d,bs", [(128, 16), (64, 32), (128, 64)])
def test_write_special_rows_and_scattered_slots(d, bs):
    g = np.random.default_rng(d + bs)
    nb, h, T = 24, 2, 150
    kx = _special_rows(g, T, h, d)
    vx = _special_rows(g, T, h, d).flip(0).contiguous()
    slots = g.permutation(nb * bs)[:T].astype(np.int64)
    slots[[7, 40, 99]] = -1
    k_gs, v_gs = 1.0 / 6.0, 0.0371
    cache = pa.nvfp4_empty_cache(nb, h, bs, d)
    pa.pa_cache_write_nvfp4(kx.cuda(), vx.cuda(), torch.from_numpy(slots).cuda(), cache,
                            k_gs, v_gs)
    torch.cuda.synchronize()
    ocache = ON.cache_write(kx.float().numpy(), vx.float().numpy(), slots,
                            ON.empty_cache(nb, h, bs, d), k_gs, v_gs)
    assert_pool_equal(cache, ocache, list(range(nb)))
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("d,bs", [(64, 16), (128, 32)])
def test_empty_and_ragged_sequences(d, bs):
    lens = [0, 1, 15, 16, 17, 0, 33, 255, 256, 257]
    w = W.Workload("ragged", len(lens), 8, 2, d, bs, seq_lens=[max(1, n) for n in lens],
                   pool_blocks=96, seed=31)
    case = build_case(w)
    case.w.seq_lens = lens
    case.lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    seqs = range(len(lens))
    snap = snapshot_blocks(case, seqs)
    k_gs, v_gs = gscales(snap)
    cache = gpu_pool(case, k_gs, v_gs)
    ocache = oracle_pool(snap, k_gs, v_gs)
    poison_unused(cache, case)
    out = run_decode(case, cache, k_gs, v_gs)
    ref = oracle_out(case, snap, ocache, k_gs, v_gs, seqs)
    assert_close(out, ref, TOL, "nvfp4 ragged")
    assert torch.equal(out[0], torch.zeros_like(out[0]))
    assert pa.pa_get_device_error() == 0


@pytest.fixture(scope="module")
def case8b():
    case = build_case(W.llama31_8b())
    seqs = list(range(0, 128, 9))
    snap = snapshot_blocks(case, seqs)
    k_gs, v_gs = gscales(snap)
    cache = gpu_pool(case, k_gs, v_gs)
    ocache = oracle_pool(snap, k_gs, v_gs)
    ref = oracle_out(case, snap, ocache, k_gs, v_gs, seqs)
    return case, cache, k_gs, v_gs, ref


@pytest.mark.parametrize("splits", [1, 2, 7, 151, 2000])
def test_partition_count_within_tolerance(case8b, splits):
    case, cache, k_gs, v_gs, ref = case8b
    out = run_decode(case, cache, k_gs, v_gs, num_splits=splits)
    assert_close(out, ref, TOL, f"nvfp4 splits={splits}")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("splits", [0, 2000])
def test_repeated_decode_is_bit_identical(case8b, splits):
    case, cache, k_gs, v_gs, _ = case8b
    outs = [run_decode(case, cache, k_gs, v_gs, num_splits=splits) for _ in range(6)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert pa.pa_get_device_error() == 0


def test_bad_table_entry_and_slot_are_flagged():
    case = build_case(W.tiny())
    cache = gpu_pool(case, 0.01, 0.01)
    tab = case.table_t.clone()
    tab[2, 1] = 10 ** 6
    out = run_decode(case, cache, 0.01, 0.01, table=tab)
    assert pa.pa_get_device_error() & pa.DEVERR_BAD_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    w = case.w
    slots = torch.tensor([3, w.pool_blocks * w.block_size + 5], dtype=torch.int64, device="cuda")
    before = [a.clone() for a in cache]
    kx = torch.ones((2, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    pa.pa_cache_write_nvfp4(kx, kx, slots, cache, 0.01, 0.01)
    assert pa.pa_get_device_error() & pa.DEVERR_BAD_SLOT
    # slot 3 (block 0, token 3) was written; nothing else changed
    assert not torch.equal(cache[0][0, :, 3], before[0][0, :, 3])
    cache[0][0, :, 3] = before[0][0, :, 3]
    cache[1][0, :, 3] = before[1][0, :, 3]
    cache[2][0, :, 1] = before[2][0, :, 1]
    cache[3][0, :, :, 3] = before[3][0, :, :, 3]
    for a, b in zip(cache, before):
        assert torch.equal(a, b)
    assert pa.pa_get_device_error() == 0


def _workload(name, B, hq, hkv, d, bs, lens, seed):
    need = sum(-(-n // bs) for n in lens)
    return W.Workload(name, B, hq, hkv, d, bs, seq_lens=lens,
                      pool_blocks=int(np.ceil(1.3 * need)) + 2, seed=seed)


def _lens(B, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


@pytest.mark.parametrize("name,B,hq,hkv,d,bs,lo,hi", [
    ("mqa", 300, 8, 1, 128, 32, 1, 600),       # several 128-sequence length scans
    ("mha_bs256", 5, 4, 4, 64, 256, 200, 1500),  # group 1, the largest block size
    ("gqa3", 40, 6, 2, 128, 16, 1, 700),       # a group of 3
    ("long1", 1, 8, 1, 64, 16, 262144, 262144),  # one 256K sequence over every CTA
])
def test_shape_parity(name, B, hq, hkv, d, bs, lo, hi):
    case = build_case(_workload(name, B, hq, hkv, d, bs, _lens(B, lo, hi, 7), 41))
    seqs = list(range(B))
    snap = snapshot_blocks(case, seqs)
    k_gs, v_gs = gscales(snap)
    cache = gpu_pool(case, k_gs, v_gs)
    ocache = oracle_pool(snap, k_gs, v_gs)
    assert_pool_equal(cache, ocache, snap[0][:256])
    poison_unused(cache, case)
    ref = oracle_out(case, snap, ocache, k_gs, v_gs, seqs)
    for splits in (0, 3):
        out = run_decode(case, cache, k_gs, v_gs, num_splits=splits)
        assert_close(out, ref, TOL, f"nvfp4 {name} splits {splits}")
    assert pa.pa_get_device_error() == 0


# ------------------------------------------------------ fused NVFP4 append --
def _fp4_two_ways(case, cache0, k_gs, v_gs, slots, splits):
    """(out, pools) of pa_cache_write_nvfp4 + pa_decode_nvfp4 and of
    pa_decode_append_nvfp4, each on its own copy of the pools."""
    w = case.w
    c1 = tuple(a.clone() for a in cache0)
    c2 = tuple(a.clone() for a in cache0)
    n = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                    splits)
    ws = torch.full((max(n, 16),), 255, dtype=torch.uint8, device="cuda")
    o1 = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"),
                    dtype=torch.bfloat16, device="cuda")
    o2 = o1.clone()
    pa.pa_cache_write_nvfp4(case.k_new, case.v_new, slots, c1, k_gs, v_gs)
    pa.pa_decode_nvfp4(case.q, c1, k_gs, v_gs, case.table_t, case.lens_t, w.scale, o1, ws,
                       num_splits=splits)
    pa.pa_decode_append_nvfp4(case.q, case.k_new, case.v_new, slots, c2, k_gs, v_gs,
                              case.table_t, case.lens_t, w.scale, o2, ws, num_splits=splits)
    torch.cuda.synchronize()
    return (o1, c1), (o2, c2)


@pytest.mark.parametrize("name", ["tiny", "llama3.2-1b", "llama3.1-8b", "shared_prefix_bs32"])
@pytest.mark.parametrize("splits", [0, 7])
def test_fused_append_equals_write_then_decode(name, splits):
    case = build_case(W.WORKLOADS[name]())
    k_gs, v_gs = 0.0029, 0.0031
    cache0 = gpu_pool(case, k_gs, v_gs)
    (o1, c1), (o2, c2) = _fp4_two_ways(case, cache0, k_gs, v_gs, case.slots_t, splits)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)), name
    for a, b in zip(c1, c2):
        assert torch.equal(a, b), name
    assert pa.pa_get_device_error() == 0


def test_fused_append_skips_and_flags_slots():
    # slot -1: nothing appended for that sequence; a slot other than the
    # last position's: flagged, not written; the rest as write-then-decode
    case = build_case(W.llama32_1b(24))
    k_gs, v_gs = 0.0029, 0.0031
    cache0 = gpu_pool(case, k_gs, v_gs)
    slots = case.slots_t.clone()
    slots[3] = -1
    good = slots.clone()
    slots[5] = slots[5] ^ 1  # the neighbouring slot of the same block
    good[5] = -1
    (o1, c1), (o2, c2) = _fp4_two_ways(case, cache0, k_gs, v_gs, slots, 0)
    err = pa.pa_get_device_error()
    assert err & pa.DEVERR_BAD_SLOT
    # the reference: write only the good slots, then decode
    (r1, rc1), _ = _fp4_two_ways(case, cache0, k_gs, v_gs, good, 0)
    pa.pa_get_device_error()
    assert torch.equal(o2.view(torch.int16), r1.view(torch.int16))
    for a, b in zip(c2, rc1):
        assert torch.equal(a, b)


def test_many_short_sequences():
    # 2048 sequences of 1..70 tokens: dozens of whole segments per CTA
    B = 2048
    case = build_case(_workload("short", B, 16, 4, 128, 16, _lens(B, 1, 70, 11), 25))
    seqs = list(range(0, B, 41))
    snap = snapshot_blocks(case, seqs)
    k_gs, v_gs = gscales(snap)
    cache = gpu_pool(case, k_gs, v_gs)
    ocache = oracle_pool(snap, k_gs, v_gs)
    assert_pool_equal(cache, ocache, snap[0][:128])
    poison_unused(cache, case)
    out = run_decode(case, cache, k_gs, v_gs)
    assert_close(out, oracle_out(case, snap, ocache, k_gs, v_gs, seqs), TOL, "nvfp4 short")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("splits", [1, 5, 37, 2000])
def test_more_partitions_than_tiles(splits):
    case = build_case(W.tiny())
    seqs = list(range(case.w.num_seqs))
    snap = snapshot_blocks(case, seqs)
    k_gs, v_gs = gscales(snap)
    cache = gpu_pool(case, k_gs, v_gs)
    ocache = oracle_pool(snap, k_gs, v_gs)
    poison_unused(cache, case)
    out = run_decode(case, cache, k_gs, v_gs, num_splits=splits)
    assert_close(out, oracle_out(case, snap, ocache, k_gs, v_gs, seqs), TOL,
                 f"nvfp4 tiny splits={splits}")
    assert pa.pa_get_device_error() == 0
