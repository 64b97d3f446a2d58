"""The bounded-wait path of the decode kernels, made to run on purpose.

Every pipeline wait in the bf16 (copy warp + math warp), FP8 head_dim 64
(single warp) and FP8 head_dim 128 (tensor-core, warp-specialised) decode
kernels gives up after a bounded number of polls, sets PA_DEVERR_TIMEOUT
and lets the CTA's own copies land before it exits.  A correct pipeline
never reaches the bound, so this test uses the test hook of
include/pa_testing.h: with stall on, every CTA's math (softmax) warps first
wait on a barrier nothing arrives at, with a short limit, so that wait runs
out deterministically (no fault, no hang: the copies the CTA issued still
land and are waited for, and the tensor-core kernel's MMA warps wait for
their MMAs before the tensor memory is released).  The call must return, the error word must carry
PA_DEVERR_TIMEOUT, and the next normal call on the same device must be
clean and match the fp64 oracle.
"""
import time

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
    yield
    pa.pa_testing_set_wait_limit(0)  # back to the default for later tests


def _ws(w, splits=0):
    n = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                    splits)
    return torch.full((max(n, 16),), 255, dtype=torch.uint8, device="cuda")


def _out(w):
    return torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"),
                      dtype=torch.bfloat16, device="cuda")


@pytest.mark.parametrize("name,splits", [("tiny", 0), ("llama3.1-8b", 0), ("llama3.1-8b", 7)])
def test_bf16_stalled_wait_times_out_then_recovers(name, splits):
    case = build_case(W.WORKLOADS[name]())
    w = case.w
    seqs = list(range(w.num_seqs)) if w.num_seqs <= 16 else list(range(0, w.num_seqs, 9))
    snap = snapshot_blocks(case, seqs)
    pa.pa_cache_write(case.k_new, case.v_new, case.slots_t, case.k_cache, case.v_cache)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    # a wait that can only run out: every CTA gives up, drains, returns
    pa.pa_testing_set_wait_limit(2000, stall=True)
    t0 = time.time()
    pa.pa_decode(case.q, case.k_cache, case.v_cache, case.table_t, case.lens_t, w.scale,
                 _out(w), _ws(w, splits), num_splits=splits)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    print(f"{name}: the stalled call returned after {elapsed:.2f} s")
    assert elapsed < 60.0
    assert pa.pa_get_device_error() & pa.DEVERR_TIMEOUT
    # the same device, normal limits: clean and correct
    pa.pa_testing_set_wait_limit(0)
    out = _out(w)
    pa.pa_decode(case.q, case.k_cache, case.v_cache, case.table_t, case.lens_t, w.scale, out,
                 _ws(w, splits), num_splits=splits)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert_close(out, oracle_decode(case, snap, seqs), 1e-2, f"{name} after a timeout")


@pytest.mark.parametrize("name", ["tiny", "llama3.1-8b"])
def test_fp8_stalled_wait_times_out_then_recovers(name):
    # tiny: head_dim 64, the single-warp kernel; the 8B shape: head_dim 128,
    # the tensor-core kernel
    case = build_case(W.WORKLOADS[name]())
    w = case.w
    seqs = list(range(w.num_seqs)) if w.num_seqs <= 16 else list(range(0, w.num_seqs, 9))
    snap = snapshot_blocks(case, seqs)
    ref, (blocks, valid, ids) = oracle_decode_fp8(case, snap, seqs)
    # an FP8 cache of the same blocks, quantised by the library
    nb, H, bs, d = case.k_cache.shape
    kq = torch.zeros((nb, H, bs, d), dtype=torch.uint8, device="cuda")
    vq = torch.zeros_like(kq)
    ks = torch.ones((nb, H), device="cuda")
    vs = torch.ones_like(ks)
    bid = torch.tensor([ids[x] for x in blocks], dtype=torch.int32, device="cuda")
    vl = torch.tensor(valid, dtype=torch.int32, device="cuda")
    pa.pa_quantize_fp8(case.k_cache, case.v_cache, bid, vl, kq, vq, ks, vs)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    pa.pa_testing_set_wait_limit(2000, stall=True)
    pa.pa_decode(case.q, kq, vq, case.table_t, case.lens_t, w.scale, _out(w), _ws(w),
                 k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() & pa.DEVERR_TIMEOUT
    pa.pa_testing_set_wait_limit(0)
    out = _out(w)
    pa.pa_decode(case.q, kq, vq, case.table_t, case.lens_t, w.scale, out, _ws(w), k_scale=ks,
                 v_scale=vs)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert_close(out, ref, 5e-2, f"{name} fp8 after a timeout")
