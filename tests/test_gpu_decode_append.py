"""GPU tests of pa_decode_append, the step's cache write and decode in one
launch: it must leave exactly the cache and the output that pa_cache_write
followed by pa_decode leave (bit for bit), and so match the fp64 oracle.

Cases cover block sizes 8 (two blocks per 16-token tile), 16 and 32, split
and unsplit segments (automatic and 7 partitions), sequences that append
nothing (slot -1), and a slot that is not where the table puts the last
position (flagged, not written).  The FP8 decode step (pa_cache_write_fp8
then pa_decode) is checked against the oracle: the cache bit for bit, the
output within the FP8 tolerance.
"""
import pytest
import torch

from paged_kv_cache_228_gb300 import pa
from paged_kv_cache_228_gb300 import workloads as W

from cases import assert_close, build_case, oracle_decode, snapshot_blocks

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_228_gb300 import build
    build.build()
    pa.pa_get_device_error()


def _workspace(w, num_splits):
    n = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                    num_splits)
    return torch.full((max(n, 16),), 255, dtype=torch.uint8, device="cuda")


def _out(w):
    return torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"),
                      dtype=torch.bfloat16, device="cuda")


def _two_ways(case, slots, num_splits):
    """(out, k, v) of write-then-decode and of the fused call, each on its
    own copy of the pool."""
    w = case.w
    k1, v1 = case.k_cache.clone(), case.v_cache.clone()
    k2, v2 = case.k_cache.clone(), case.v_cache.clone()
    o1, o2 = _out(w), _out(w)
    pa.pa_cache_write(case.k_new, case.v_new, slots, k1, v1)
    pa.pa_decode(case.q, k1, v1, case.table_t, case.lens_t, w.scale, o1,
                 _workspace(w, num_splits), num_splits=num_splits)
    pa.pa_decode_append(case.q, case.k_new, case.v_new, slots, k2, v2, case.table_t,
                        case.lens_t, w.scale, o2, _workspace(w, num_splits),
                        num_splits=num_splits)
    torch.cuda.synchronize()
    return (o1, k1, v1), (o2, k2, v2)


def _bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("name", ["tiny", "llama3.2-1b", "llama3.1-8b", "shared_prefix_bs8",
                                  "shared_prefix_bs32"])
@pytest.mark.parametrize("splits", [0, 7])
def test_fused_equals_write_then_decode(name, splits):
    case = build_case(W.WORKLOADS[name]())
    (o1, k1, v1), (o2, k2, v2) = _two_ways(case, case.slots_t, splits)
    assert torch.equal(_bits(o1), _bits(o2)), name
    assert torch.equal(_bits(k1), _bits(k2)) and torch.equal(_bits(v1), _bits(v2)), name
    assert pa.pa_get_device_error() == 0


def test_fused_matches_oracle():
    case = build_case(W.llama31_8b(), poison_unused=True)
    seqs = range(case.w.num_seqs)
    snap = snapshot_blocks(case, seqs)
    w = case.w
    out = _out(w)
    pa.pa_decode_append(case.q, case.k_new, case.v_new, case.slots_t, case.k_cache,
                        case.v_cache, case.table_t, case.lens_t, w.scale, out,
                        _workspace(w, 0))
    torch.cuda.synchronize()
    assert_close(out, oracle_decode(case, snap, seqs), TOL_BF16, "fused append 8B")
    assert pa.pa_get_device_error() == 0


def test_sequences_without_append():
    # slot -1: the sequence appends nothing; position n - 1 keeps what the
    # pool held, in both ways of running the step
    case = build_case(W.llama32_1b())
    slots = case.slots_t.clone()
    slots[::3] = -1
    (o1, k1, v1), (o2, k2, v2) = _two_ways(case, slots, 0)
    assert torch.equal(_bits(o1), _bits(o2))
    assert torch.equal(_bits(k1), _bits(k2)) and torch.equal(_bits(v1), _bits(v2))
    assert pa.pa_get_device_error() == 0


def test_misplaced_slot_is_flagged_and_not_written():
    case = build_case(W.tiny())
    w = case.w
    slots = case.slots_t.clone()
    slots[1] = slots[1] - 1          # a slot, but not position n - 1's
    k2, v2 = case.k_cache.clone(), case.v_cache.clone()
    before_k = k2.clone()
    pa.pa_decode_append(case.q, case.k_new, case.v_new, slots, k2, v2, case.table_t,
                        case.lens_t, w.scale, _out(w), _workspace(w, 0))
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() & pa.DEVERR_BAD_SLOT
    s = int(case.slots[1]) - 1
    blk, off = s // w.block_size, s % w.block_size
    assert torch.equal(_bits(k2[blk, :, off]), _bits(before_k[blk, :, off]))
    # the other sequences still appended
    s0 = int(case.slots[0])
    assert torch.equal(_bits(k2[s0 // w.block_size, :, s0 % w.block_size]),
                       _bits(case.k_new[0]))


# ------------------------------------------------- FP8 step: append+decode ---
@pytest.mark.parametrize("name", ["tiny", "llama3.1-8b", "shared_prefix_bs8"])
def test_fp8_append_then_decode_matches_oracle(name):
    # The FP8 decode step: the pre-step cache is the oracle's whole-block
    # quantisation of each block's valid tokens; pa_cache_write_fp8 appends
    # the step's tokens (grow-only scales), pa_decode reads the result.
    import numpy as np
    from oracle import paged_attention as OPA
    from oracle import quantize as OQ
    from cases import _to_np32, _to_np64

    case = build_case(W.WORKLOADS[name]())
    w = case.w
    bs = w.block_size
    seqs = list(range(w.num_seqs)) if w.num_seqs <= 128 else list(range(0, w.num_seqs, 8))
    ids, kk, vv = snapshot_blocks(case, range(w.num_seqs))
    local = {bid: i for i, bid in enumerate(ids)}
    valid = {}
    for b in range(w.num_seqs):
        n0 = w.seq_lens[b] - 1                       # before the append
        for j, x in enumerate(case.tables[b]):
            valid[local[x]] = max(valid.get(local[x], 0), max(0, min(bs, n0 - j * bs)))
    blocks = sorted(valid)
    kq, ks = OQ.quantize_blocks(kk, blocks, [valid[x] for x in blocks])
    vq, vs = OQ.quantize_blocks(vv, blocks, [valid[x] for x in blocks])

    dev = "cuda"
    shape = (w.pool_blocks, w.num_kv_heads, bs, w.head_dim)
    gk = torch.zeros(shape, dtype=torch.uint8, device=dev)
    gv = torch.zeros_like(gk)
    gks = torch.ones((w.pool_blocks, w.num_kv_heads), device=dev)
    gvs = torch.ones_like(gks)
    idx = torch.tensor(ids, dtype=torch.int64, device=dev)
    gk[idx], gv[idx] = torch.from_numpy(kq).to(dev), torch.from_numpy(vq).to(dev)
    gks[idx], gvs[idx] = torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev)
    out = _out(w)
    pa.pa_cache_write_fp8(case.k_new, case.v_new, case.slots_t, gk, gv, gks, gvs)
    pa.pa_decode(case.q, gk, gv, case.table_t, case.lens_t, w.scale, out, _workspace(w, 0),
                 k_scale=gks, v_scale=gvs)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0

    sl = np.array([local[s // bs] * bs + s % bs for s in case.slots], dtype=np.int64)
    kq2, vq2, ks2, vs2 = OQ.cache_write_fp8(_to_np32(case.k_new), _to_np32(case.v_new), sl,
                                            kq, vq, ks, vs)
    # the cache the kernel left equals the oracle's, bit for bit
    assert np.array_equal(gk[idx].cpu().numpy(), kq2) and np.array_equal(gv[idx].cpu().numpy(), vq2)
    assert np.array_equal(gks[idx].cpu().numpy(), ks2) and np.array_equal(gvs[idx].cpu().numpy(), vs2)
    tab = -np.ones((w.num_seqs, max(len(t) for t in case.tables)), dtype=np.int64)
    for b in range(w.num_seqs):
        tab[b, :len(case.tables[b])] = [local[x] for x in case.tables[b]]
    ref = OPA.decode(_to_np64(case.q), kq2, vq2, tab, np.array(w.seq_lens), w.scale,
                     k_scale=ks2, v_scale=vs2, seqs=seqs)
    assert_close(out, ref, 5e-2, f"{name} fp8 append+decode")


@pytest.mark.parametrize("name,splits", [("llama3.1-8b", 0), ("llama3.1-8b", 7),
                                         ("shared_prefix_bs8", 0), ("tiny", 0)])
def test_fp8_fused_equals_write_then_decode(name, splits):
    # pa_decode_append_fp8 against pa_cache_write_fp8 + pa_decode on copies
    # of one FP8 cache: codes, scales and output bit for bit.  Half the new
    # tokens are scaled up so that their blocks' scales grow.
    import numpy as np
    from oracle import quantize as OQ
    case = build_case(W.WORKLOADS[name]())
    w = case.w
    ids, kk, vv = snapshot_blocks(case, range(w.num_seqs))
    valid = {}
    local = {bid: i for i, bid in enumerate(ids)}
    for b in range(w.num_seqs):
        n0 = w.seq_lens[b] - 1
        for j, x in enumerate(case.tables[b]):
            valid[local[x]] = max(valid.get(local[x], 0), max(0, min(w.block_size, n0 - j * w.block_size)))
    blocks = sorted(valid)
    kq, ks = OQ.quantize_blocks(kk, blocks, [valid[x] for x in blocks])
    vq, vs = OQ.quantize_blocks(vv, blocks, [valid[x] for x in blocks])
    shape = (w.pool_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    idx = torch.tensor(ids, dtype=torch.int64, device="cuda")

    def pool():
        k = torch.zeros(shape, dtype=torch.uint8, device="cuda")
        v = torch.zeros_like(k)
        s1 = torch.ones((w.pool_blocks, w.num_kv_heads), device="cuda")
        s2 = torch.ones_like(s1)
        k[idx], v[idx] = torch.from_numpy(kq).cuda(), torch.from_numpy(vq).cuda()
        s1[idx], s2[idx] = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
        return k, v, s1, s2

    grow = torch.ones((w.num_seqs, 1, 1), device="cuda")
    grow[::2] = 25.0
    kn = (case.k_new.float() * grow).to(torch.bfloat16)
    vn = (case.v_new.float() * grow).to(torch.bfloat16)
    k1, v1, ks1, vs1 = pool()
    k2, v2, ks2, vs2 = pool()
    o1, o2 = _out(w), _out(w)
    pa.pa_cache_write_fp8(kn, vn, case.slots_t, k1, v1, ks1, vs1)
    pa.pa_decode(case.q, k1, v1, case.table_t, case.lens_t, w.scale, o1, _workspace(w, splits),
                 k_scale=ks1, v_scale=vs1, num_splits=splits)
    pa.pa_decode_append_fp8(case.q, kn, vn, case.slots_t, k2, v2, ks2, vs2, case.table_t,
                            case.lens_t, w.scale, o2, _workspace(w, splits), num_splits=splits)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert torch.equal(k1, k2) and torch.equal(v1, v2), name
    assert torch.equal(ks1, ks2) and torch.equal(vs1, vs2), name
    assert torch.equal(_bits(o1), _bits(o2)), name


def test_fp8_fused_rejects_large_blocks():
    case = build_case(W.shared_prefix(32, num_seqs=4, prefix=64))
    w = case.w
    k = torch.zeros(case.k_cache.shape, dtype=torch.uint8, device="cuda")
    s = torch.ones((w.pool_blocks, w.num_kv_heads), device="cuda")
    with pytest.raises(RuntimeError):
        pa.pa_decode_append_fp8(case.q, case.k_new, case.v_new, case.slots_t, k, k.clone(), s,
                                s.clone(), case.table_t, case.lens_t, w.scale, _out(w),
                                _workspace(w, 0))
