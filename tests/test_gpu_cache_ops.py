"""GPU parity of the cache kernels against the oracle, bit for bit.

* pa_cache_write: every config's append step, plus random distinct slots
  with skipped (negative) slots, for bs in {8, 16, 32} and d in {64, 128};
* pa_copy_blocks: copy-on-write pairs from a real fork, bf16 and FP8 (with
  scales);
* pa_quantize_fp8: codes and scales equal the oracle's quantiser (its own
  E4M3 encoder), including outlier-heavy and partially valid blocks; a
  cross-check of a sample of codes against torch's float8_e4m3fn cast.
"""
import numpy as np
import pytest
import torch

from oracle import e2m1, e4m3
from oracle import paged_attention as OPA
from oracle import quantize as OQ
from paged_kv_cache_228_gb300 import pa
from paged_kv_cache_228_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_228_gb300 import build
    build.build()
    pa.pa_get_device_error()  # clear


def _bits(t):
    return t.detach().cpu().view(torch.int16 if t.element_size() == 2 else torch.uint8).numpy()


@pytest.mark.parametrize("bs,d,nb,H,T", [(16, 64, 32, 2, 4), (8, 128, 64, 8, 37),
                                         (32, 128, 40, 8, 128), (16, 128, 300, 8, 256)])
def test_cache_write_bit_exact(bs, d, nb, H, T):
    dev = "cuda"
    kc = W.normal_bf16((nb, H, bs, d), 11, dev)
    vc = W.normal_bf16((nb, H, bs, d), 12, dev)
    kn = W.normal_bf16((T, H, d), 13, dev)
    vn = W.normal_bf16((T, H, d), 14, dev)
    slots = W.distinct_slots(nb * bs, T, 15)
    slots[::5] = -1
    ek, ev = OPA.cache_write(_bits(kn), _bits(vn), slots.numpy(), _bits(kc), _bits(vc))
    pa.pa_cache_write(kn, vn, slots.to(dev), kc, vc)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kc), ek)
    assert np.array_equal(_bits(vc), ev)
    assert pa.pa_get_device_error() == 0


def test_cache_write_bad_slot_is_flagged_and_skipped():
    dev = "cuda"
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    kn = torch.ones((2, 2, 64), dtype=torch.bfloat16, device=dev)
    slots = torch.tensor([3, 4 * 16 + 5], dtype=torch.int64, device=dev)
    pa.pa_cache_write(kn, kn, slots, kc, vc)
    assert pa.pa_get_device_error() & pa.DEVERR_BAD_SLOT
    assert kc.sum().item() == 2 * 64  # only slot 3 written
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_copy_blocks_bit_exact(fp8):
    dev = "cuda"
    nb, H, bs, d = 24, 4, 16, 128
    if fp8:
        kc = torch.randint(0, 255, (nb, H, bs, d), dtype=torch.uint8, device=dev)
        vc = torch.randint(0, 255, (nb, H, bs, d), dtype=torch.uint8, device=dev)
        ks = torch.rand((nb, H), device=dev)
        vs = torch.rand((nb, H), device=dev)
    else:
        kc = W.normal_bf16((nb, H, bs, d), 21, dev)
        vc = W.normal_bf16((nb, H, bs, d), 22, dev)
        ks = vs = None
    # a real fork: parent of 2 * 16 + 5 tokens, three children append one token
    a = pa.Allocator(nb)
    parent = []
    a.append_slots(parent, 0, 37, bs, 8)
    pairs = []
    for _ in range(3):
        child = list(parent)
        a.fork(child)
        st, _, pr = a.append_slots(child, 37, 1, bs, 8)
        pairs += pr
    assert len(pairs) == 3 and all(p[2] == 5 for p in pairs)
    ek, ev = OPA.copy_blocks(_bits(kc), _bits(vc), pairs)
    pa.pa_copy_blocks(kc, vc, torch.tensor(pairs, dtype=torch.int32, device=dev), ks, vs)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kc), ek) and np.array_equal(_bits(vc), ev)
    if fp8:
        for s, dd, _ in pairs:
            assert torch.equal(ks[dd], ks[s]) and torch.equal(vs[dd], vs[s])
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("bs,d", [(16, 128), (8, 64), (32, 128)])
def test_quantize_fp8_bit_exact(bs, d):
    dev = "cuda"
    nb, H = 40, 4
    k = W.normal_bf16((nb, H, bs, d), 31, dev, outlier_prob=0.01, outlier_scale=20.0)
    v = W.normal_bf16((nb, H, bs, d), 32, dev, outlier_prob=0.01, outlier_scale=20.0)
    k[3] = 0  # an all-zero block: scale 1
    ids = [3, 7, 0, 39, 12, 5]
    valid = [bs, bs, 1, bs // 2, bs - 1, 0]
    kq = torch.full((nb, H, bs, d), 0xAB, dtype=torch.uint8, device=dev)
    vq = torch.full_like(kq, 0xCD)
    ks = torch.full((nb, H), -1.0, device=dev)
    vs = torch.full((nb, H), -1.0, device=dev)
    pa.pa_quantize_fp8(k, v, torch.tensor(ids, dtype=torch.int32, device=dev),
                       torch.tensor(valid, dtype=torch.int32, device=dev), kq, vq, ks, vs)
    torch.cuda.synchronize()
    k32 = k.float().cpu().numpy()
    v32 = v.float().cpu().numpy()
    eq, es = OQ.quantize_blocks(k32, ids, valid)
    fq, fs = OQ.quantize_blocks(v32, ids, valid)
    for i in ids:
        assert np.array_equal(kq[i].cpu().numpy(), eq[i]), i
        assert np.array_equal(vq[i].cpu().numpy(), fq[i]), i
        assert np.array_equal(ks[i].cpu().numpy(), es[i]), i
        assert np.array_equal(vs[i].cpu().numpy(), fs[i]), i
    # untouched blocks keep their contents
    assert (kq[1] == 0xAB).all() and (ks[1] == -1).all()
    assert pa.pa_get_device_error() == 0


def test_quantize_codes_agree_with_torch_cast():
    # Library cross-check of the GPU conversion (inside +-448 torch's cast
    # is RNE like the kernel's satfinite conversion).
    dev = "cuda"
    k = W.normal_bf16((8, 2, 16, 128), 41, dev)
    ids = torch.arange(8, dtype=torch.int32, device=dev)
    valid = torch.full((8,), 16, dtype=torch.int32, device=dev)
    kq = torch.empty((8, 2, 16, 128), dtype=torch.uint8, device=dev)
    ks = torch.empty((8, 2), device=dev)
    pa.pa_quantize_fp8(k, k, ids, valid, kq, kq.clone(), ks, ks.clone())
    kc = k.float().cpu()
    s = kc.abs().amax(dim=(2, 3)) / torch.tensor(448.0)  # fp32 IEEE on the CPU
    x = kc / s[:, :, None, None]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(ref, kq.cpu())


# ------------------------------------------------------------ FP8 append ---
def _fp8_pool(nb, H, bs, d, fill, seed, dev="cuda"):
    """An FP8 pool whose blocks [0, nb) hold `fill[b]` valid tokens, built by
    the oracle's whole-block quantiser from seeded bf16 values (outliers
    included), with stale bytes past each fill."""
    x = W.normal_bf16((nb, H, bs, d), seed, "cpu", outlier_prob=0.01, outlier_scale=20.0)
    codes, scales = OQ.quantize_blocks(x.float().numpy(), list(range(nb)), fill)
    for b, n in enumerate(fill):
        codes[b, :, n:] = 0x3C          # stale bytes a reused block may hold
    return (torch.from_numpy(codes).to(dev), torch.from_numpy(scales).to(dev))


@pytest.mark.parametrize("bs,d", [(16, 128), (8, 64), (32, 128), (16, 64)])
def test_cache_write_fp8_bit_exact(bs, d):
    # Several steps of one appended token per sequence, each sequence in its
    # own block: fresh blocks (offset 0), appends under the current scale
    # and appends that grow it (outlier tokens), against the oracle.
    dev = "cuda"
    nb, H, T = 24, 4, 20
    g = np.random.default_rng(bs * 1000 + d)
    fill = [int(x) for x in g.integers(0, bs - 3, size=nb)]
    kq, ks = _fp8_pool(nb, H, bs, d, fill, 51)
    vq, vs = _fp8_pool(nb, H, bs, d, fill, 52)
    blocks = g.permutation(nb)[:T]
    ref = [kq.cpu().numpy(), vq.cpu().numpy(), ks.cpu().numpy(), vs.cpu().numpy()]
    for step in range(3):
        scale = torch.ones((T, H, 1))
        scale[::3] = 30.0               # these tokens raise their block's scale
        kn = (W.normal_bf16((T, H, d), 60 + step).float() * scale).to(torch.bfloat16)
        vn = (W.normal_bf16((T, H, d), 70 + step).float() * scale).to(torch.bfloat16)
        slots = np.array([b * bs + fill[b] + step for b in blocks], dtype=np.int64)
        slots[5] = -1                    # skipped
        pa.pa_cache_write_fp8(kn.to(dev), vn.to(dev), torch.from_numpy(slots).to(dev),
                              kq, vq, ks, vs)
        ref = list(OQ.cache_write_fp8(kn.float().numpy(), vn.float().numpy(), slots, *ref))
    torch.cuda.synchronize()
    assert np.array_equal(kq.cpu().numpy(), ref[0])
    assert np.array_equal(vq.cpu().numpy(), ref[1])
    assert np.array_equal(ks.cpu().numpy(), ref[2])
    assert np.array_equal(vs.cpu().numpy(), ref[3])
    assert pa.pa_get_device_error() == 0


def test_cache_write_fp8_bad_slot_is_flagged_and_skipped():
    dev = "cuda"
    kq, ks = _fp8_pool(4, 2, 16, 64, [3] * 4, 81)
    vq, vs = _fp8_pool(4, 2, 16, 64, [3] * 4, 82)
    k0, s0 = kq.clone(), ks.clone()
    kn = W.normal_bf16((2, 2, 64), 83).to(dev)
    pa.pa_cache_write_fp8(kn, kn, torch.tensor([4 * 16, -5], dtype=torch.int64, device=dev),
                          kq, vq, ks, vs)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() & pa.DEVERR_BAD_SLOT
    assert torch.equal(kq, k0) and torch.equal(ks, s0)


def _bf16_values(limit):
    """Every finite bf16 value with |x| <= limit, as float32 (both zeros)."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).float()
    keep = torch.isfinite(x) & (x.abs() <= limit)
    return x[keep]


def test_quantize_codes_exhaustive_over_bf16():
    # Every bf16 input in [-448, 448] through the GPU conversion: each (block,
    # head) tile holds one 448, so its scale is exactly 1 and the code is
    # e4m3(x); the oracle encodes the same values.
    dev = "cuda"
    vals = _bf16_values(448.0)
    per = 16 * 128 - 1
    n_tiles = -(-vals.numel() // per)
    x = torch.zeros(n_tiles * per)
    x[:vals.numel()] = vals
    tiles = torch.cat([torch.full((n_tiles, 1), 448.0), x.view(n_tiles, per)], dim=1)
    k = tiles.view(n_tiles, 1, 16, 128).to(torch.bfloat16).to(dev)
    ids = torch.arange(n_tiles, dtype=torch.int32, device=dev)
    valid = torch.full((n_tiles,), 16, dtype=torch.int32, device=dev)
    kq = torch.empty(k.shape, dtype=torch.uint8, device=dev)
    ks = torch.empty((n_tiles, 1), device=dev)
    pa.pa_quantize_fp8(k, k, ids, valid, kq, kq.clone(), ks, ks.clone())
    torch.cuda.synchronize()
    assert torch.all(ks == 1.0)
    got = kq.view(n_tiles, -1)[:, 1:].reshape(-1)[:vals.numel()].cpu().numpy()
    ref = e4m3.encode_fast(vals.numpy())
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, (bad.size, vals[bad[:5]].tolist(), got[bad[:5]], ref[bad[:5]])
    assert pa.pa_get_device_error() == 0


def test_nvfp4_codes_exhaustive_over_bf16():
    # Every bf16 input in [-6, 6] through the NVFP4 writer: each 16-value
    # group holds one 6 and the tensor scale is 1/6, so the block scale is 6
    # (E4M3 0x4C), the divisor 6 * (1/6) rounds to exactly 1 in fp32, and the
    # code is e2m1(x); the oracle encodes the same values.
    dev = "cuda"
    vals = _bf16_values(6.0)
    per_row = 128 - 8                                 # 8 groups of 15 values + one 6
    rows = -(-vals.numel() // per_row)
    x = torch.zeros(rows * per_row)
    x[:vals.numel()] = vals
    g = x.view(rows, 8, 15)
    row = torch.cat([torch.full((rows, 8, 1), 6.0), g], dim=2).view(rows, 1, 128)
    kn = row.to(torch.bfloat16).to(dev)
    bs = 16
    nb = -(-rows // bs)
    cache = pa.nvfp4_empty_cache(nb, 1, bs, 128)
    slots = torch.arange(rows, dtype=torch.int64, device=dev)
    pa.pa_cache_write_nvfp4(kn, kn, slots, cache, 1.0 / 6.0, 1.0 / 6.0)
    torch.cuda.synchronize()
    k, k_sf = cache[0].cpu().numpy(), cache[1].cpu().numpy()
    assert np.all(k_sf.reshape(-1)[:rows * 8] == 0x4C)
    b = k.reshape(nb * bs, 64)[:rows]
    codes = np.stack([b & 0xF, b >> 4], axis=-1).reshape(rows, 8, 16)[:, :, 1:]
    got = codes.reshape(-1)[:vals.numel()]
    ref = e2m1.encode(vals.numpy())
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, (bad.size, vals[bad[:5]].tolist(), got[bad[:5]], ref[bad[:5]])
    assert pa.pa_get_device_error() == 0
