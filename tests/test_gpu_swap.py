"""GPU tests of pa_swap_out / pa_swap_in (cache blocks to pinned host memory
and back, read and written in place by the kernel): bit for bit against
plain indexing of the pool's CPU copy, bf16 and FP8 (with scales), block
sizes 8 and 16, and an id outside the pool (flagged, skipped)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_228_gb300 import pa
from paged_kv_cache_228_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_228_gb300 import build
    build.build()
    pa.pa_get_device_error()


def _bits(t):
    return t.view(torch.uint8).numpy()


@pytest.mark.parametrize("fp8,bs,d", [(False, 16, 128), (False, 8, 64), (True, 16, 128),
                                      (True, 8, 64)])
def test_swap_round_trip(fp8, bs, d):
    nb, H = 40, 4
    k = W.normal_bf16((nb, H, bs, d), 91, "cuda")
    v = W.normal_bf16((nb, H, bs, d), 92, "cuda")
    ks = vs = None
    if fp8:
        kq = torch.empty((nb, H, bs, d), dtype=torch.uint8, device="cuda")
        vq = torch.empty_like(kq)
        ks = torch.empty((nb, H), device="cuda")
        vs = torch.empty_like(ks)
        ids = torch.arange(nb, dtype=torch.int32, device="cuda")
        pa.pa_quantize_fp8(k, v, ids, torch.full((nb,), bs, dtype=torch.int32, device="cuda"),
                           kq, vq, ks, vs)
        k, v = kq, vq
    kc, vc = k.cpu(), v.cpu()                       # the expected values come from here
    sel = [7, 0, 39, 12, 12, 25]
    ids = torch.tensor(sel, dtype=torch.int32, device="cuda")
    hk = torch.empty((len(sel), H, bs, d), dtype=k.dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    hks = torch.empty((len(sel), H)).pin_memory() if fp8 else None
    hvs = torch.empty((len(sel), H)).pin_memory() if fp8 else None
    pa.pa_swap_out(k, v, ids, hk, hv, ks, vs, hks, hvs)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(hk), _bits(kc[sel])) and np.array_equal(_bits(hv), _bits(vc[sel]))
    if fp8:
        assert torch.equal(hks, ks.cpu()[sel]) and torch.equal(hvs, vs.cpu()[sel])
    # back into other blocks of a zeroed pool
    dst = [3, 4, 5, 6, 20, 21]
    k2, v2 = torch.zeros_like(k), torch.zeros_like(v)
    ks2 = torch.zeros_like(ks) if fp8 else None
    vs2 = torch.zeros_like(vs) if fp8 else None
    pa.pa_swap_in(hk, hv, torch.tensor(dst, dtype=torch.int32, device="cuda"), k2, v2,
                  hks, hvs, ks2, vs2)
    torch.cuda.synchronize()
    k2c, v2c = k2.cpu(), v2.cpu()
    assert np.array_equal(_bits(k2c[dst]), _bits(kc[sel]))
    assert np.array_equal(_bits(v2c[dst]), _bits(vc[sel]))
    rest = [i for i in range(nb) if i not in dst]
    assert not _bits(k2c[rest]).any() and not _bits(v2c[rest]).any()
    if fp8:
        assert torch.equal(ks2.cpu()[dst], ks.cpu()[sel])
    assert pa.pa_get_device_error() == 0


def test_swap_bad_id_is_flagged_and_skipped():
    k = W.normal_bf16((8, 2, 16, 64), 93, "cuda")
    hk = torch.zeros((2, 2, 16, 64), dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    pa.pa_swap_out(k, k, torch.tensor([1, 8], dtype=torch.int32, device="cuda"), hk, hv)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() & pa.DEVERR_BAD_BLOCK_ID
    assert torch.equal(hk[0].view(torch.int16), k[1].cpu().view(torch.int16))
    assert not hk[1].view(torch.int16).any()


def test_swap_rejects_pageable_host_memory():
    k = W.normal_bf16((4, 2, 16, 64), 94, "cuda")
    hk = torch.zeros((1, 2, 16, 64), dtype=torch.bfloat16)      # not pinned
    with pytest.raises(RuntimeError):
        pa.pa_swap_out(k, k, torch.tensor([0], dtype=torch.int32, device="cuda"), hk, hk)
