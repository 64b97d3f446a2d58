"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc -- plugin hosts that
forbid allocation inside their execute callback, services that fix their
device-memory budget at start-up, thin foreign-function callers without a
device allocator.  For them the library keeps its own fixed device array
(16 MiB) as decode scratch.  These tests call that entry point through the
C ABI and compare it with pa_decode given a caller-allocated workspace,
within the bf16 decode tolerance, on two calls in a row with different
shapes (the second call runs over whatever the first left in the shared
array), and check that a shape needing more scratch than the array holds
is refused.  The file is named to run last, and passes alone or after the
other tests.
"""
import ctypes

import pytest
import torch

from paged_kv_cache_228_gb300 import pa
from paged_kv_cache_228_gb300 import workloads as W

from cases import build_case

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_228_gb300 import build
    build.build()
    pa.pa_get_device_error()


def _with_workspace(case):
    w = case.w
    n = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim)
    ws = torch.full((max(n, 16),), 255, dtype=torch.uint8, device="cuda")
    out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.bfloat16,
                      device="cuda")
    pa.pa_decode(case.q, case.k_cache, case.v_cache, case.table_t, case.lens_t, w.scale,
                 out, ws)
    return out


def _noalloc_raw(case, num_splits=0):
    """Direct C-ABI call of pa_decode_noalloc (no Python wrapper)."""
    w = case.w
    out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"),
                     dtype=torch.bfloat16, device="cuda")
    vp = ctypes.c_void_p
    st = pa.lib().pa_decode_noalloc(
        vp(case.q.data_ptr()), vp(case.k_cache.data_ptr()), vp(case.v_cache.data_ptr()),
        None, None, pa.PA_KV_BF16, vp(case.table_t.data_ptr()), case.table_t.shape[1],
        vp(case.lens_t.data_ptr()), w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
        w.block_size, w.pool_blocks, ctypes.c_float(w.scale), vp(out.data_ptr()),
        num_splits, vp(torch.cuda.current_stream().cuda_stream))
    return st, out


def _check_close(a, b):
    a64, b64 = a.double(), b.double()
    assert torch.isfinite(a64).all()
    assert ((a64 - b64).abs() <= TOL_BF16 + TOL_BF16 * b64.abs()).all()


def test_noalloc_matches_workspace_decode_on_two_calls():
    first = build_case(W.llama31_8b())       # split pieces: the scratch is used
    second = build_case(W.llama32_1b())      # different shape on the same scratch
    for case in (first, second):
        ref = _with_workspace(case)
        st, out = _noalloc_raw(case)
        assert st == pa.PA_OK, pa.status_string(st)
        torch.cuda.synchronize()
        _check_close(out, ref)
    # and once more through the binding, after the second shape
    w = first.w
    out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.bfloat16,
                      device="cuda")
    pa.pa_decode_noalloc(first.q, first.k_cache, first.v_cache, first.table_t,
                         first.lens_t, first.w.scale, out)
    torch.cuda.synchronize()
    _check_close(out, _with_workspace(first))
    assert pa.pa_get_device_error() == 0


def test_noalloc_rejects_requests_beyond_its_scratch():
    # 5000 work partitions at d = 128 need more than 16 MiB of partials
    case = build_case(W.llama31_8b())
    w = case.w
    need = pa.pa_decode_workspace_size(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                       5000)
    assert need > pa.NOALLOC_SCRATCH_BYTES
    st, out = _noalloc_raw(case, num_splits=5000)
    assert st == pa.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()      # nothing was enqueued
