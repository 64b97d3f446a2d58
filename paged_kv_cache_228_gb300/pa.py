"""Python binding of libpa (argument marshalling only).

Every function here forwards to the C ABI declared in ``include/pa.h`` under
the same name; torch tensors are used only as device (or host) memory and
their current CUDA stream.  No computation of the method happens in Python:
if ``libpa.so`` is missing, importing the functions raises instead of
falling back to anything else.

Ordering of ``seq_lens``: every decode call (pa_decode*, pa_decode_cascade,
pa_decode_noalloc) launches as a programmatic dependent of the work before
it on the stream and reads ``seq_lens`` to split its work BEFORE it waits
for that work.  Nothing in this library writes ``seq_lens``.  If a kernel of
yours writes ``seq_lens`` and calls ``griddepcontrol.launch_dependents``
(lets its dependents start early), do not launch a decode call directly
after it on the same stream: put a copy or any kernel
without that trigger in between.  Ordinary stream order (torch ops, copies)
needs nothing.
"""
from __future__ import annotations

import ctypes
import itertools
import os
import time

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_OUT_OF_BLOCKS, PA_ERR_BAD_BLOCK_ID = 0, 1, 2, 3
PA_ERR_CUDA, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE = 4, 5, 6
PA_KV_BF16, PA_KV_FP8_E4M3, PA_KV_NVFP4 = 0, 1, 2

DEVERR_BAD_BLOCK_ID, DEVERR_BAD_SEQ_LEN, DEVERR_BAD_SLOT = 0x1, 0x2, 0x4
DEVERR_BAD_PAIR, DEVERR_TIMEOUT, DEVERR_LAUNCH = 0x8, 0x10, 0x20

_lib = None

_c_int = ctypes.c_int32
_c_ptr = ctypes.c_void_p
_c_size = ctypes.c_size_t

# name -> (restype, argtypes); must match include/pa.h
SIGNATURES = {
    "pa_abi_version": (_c_int, []),
    "pa_testing_set_wait_limit": (_c_int, [ctypes.c_uint32, _c_int]),
    "pa_status_string": (ctypes.c_char_p, [_c_int]),
    "pa_get_device_error": (_c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "pa_cache_write": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_int,
                                _c_int, _c_int, _c_int, _c_int, _c_ptr]),
    "pa_cache_write_fp8": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_ptr,
                                    _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_ptr]),
    "pa_swap_out": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr,
                             _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int, _c_ptr]),
    "pa_swap_in": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr,
                            _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int, _c_ptr]),
    "pa_copy_blocks": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_int,
                                _c_int, _c_int, _c_int, _c_int, _c_ptr]),
    "pa_quantize_fp8": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr,
                                 _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_ptr]),
    "pa_decode_workspace_size": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int,
                                          ctypes.POINTER(_c_size)]),
    "pa_decode": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_int,
                           _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                           ctypes.c_float, _c_ptr, _c_ptr, _c_size, _c_int, _c_ptr]),
    "pa_decode_append": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                  _c_int, _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int,
                                  _c_int, ctypes.c_float, _c_ptr, _c_ptr, _c_size, _c_int,
                                  _c_ptr]),
    "pa_decode_cascade_workspace_size": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int,
                                                  _c_int, _c_int, ctypes.POINTER(_c_size)]),
    "pa_decode_cascade": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_int,
                                   _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                   ctypes.c_float, _c_ptr, _c_ptr, _c_size, _c_int, _c_ptr]),
    "pa_decode_append_fp8": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                      _c_ptr, _c_ptr, _c_int, _c_ptr, _c_int, _c_int, _c_int,
                                      _c_int, _c_int, _c_int, ctypes.c_float, _c_ptr, _c_ptr,
                                      _c_size, _c_int, _c_ptr]),
    "pa_decode_noalloc": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr,
                                   _c_int, _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int,
                                   _c_int, ctypes.c_float, _c_ptr, _c_int, _c_ptr]),
    "pa_cache_write_nvfp4": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_ptr,
                                      _c_ptr, ctypes.c_float, ctypes.c_float, _c_int, _c_int,
                                      _c_int, _c_int, _c_ptr]),
    "pa_decode_nvfp4": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, ctypes.c_float,
                                 ctypes.c_float, _c_ptr, _c_int, _c_ptr, _c_int, _c_int, _c_int,
                                 _c_int, _c_int, _c_int, ctypes.c_float, _c_ptr, _c_ptr,
                                 _c_size, _c_int, _c_ptr]),
    "pa_decode_append_nvfp4": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                        _c_ptr, ctypes.c_float, ctypes.c_float, _c_ptr, _c_int,
                                        _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                        ctypes.c_float, _c_ptr, _c_ptr, _c_size, _c_int,
                                        _c_ptr]),
    "pa_allocator_create": (_c_int, [_c_int, ctypes.POINTER(_c_ptr)]),
    "pa_allocator_destroy": (None, [_c_ptr]),
    "pa_block_alloc": (_c_int, [_c_ptr, _c_int, _c_ptr]),
    "pa_block_free": (_c_int, [_c_ptr, _c_ptr, _c_int]),
    "pa_block_fork": (_c_int, [_c_ptr, _c_ptr, _c_int]),
    "pa_block_refcount": (_c_int, [_c_ptr, _c_int, ctypes.POINTER(_c_int)]),
    "pa_block_num_free": (_c_int, [_c_ptr]),
    "pa_seq_append_slots": (_c_int, [_c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int,
                                     _c_ptr, _c_ptr, ctypes.POINTER(_c_int)]),
    "pa_allocator_usage": (_c_int, [_c_ptr, _c_ptr, _c_int, _c_ptr, _c_int, _c_int, _c_ptr]),
    "pa_batch_append_slots": (_c_int, [_c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_int, _c_int,
                                       _c_ptr, _c_ptr, _c_ptr, ctypes.POINTER(_c_int)]),
}


class PAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """The loaded libpa; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m paged_kv_cache_228_gb300.build` (there is no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pa_status_string(status).decode()


def _check(fn: str, status: int):
    if status != PA_OK:
        raise PAError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need(t, dtype, name, ndim=None):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got {t.dim()}")


def _kv_dtype(cache):
    if cache.dtype == torch.bfloat16:
        return PA_KV_BF16
    if cache.dtype in (torch.uint8, torch.float8_e4m3fn):
        return PA_KV_FP8_E4M3
    raise TypeError(f"unsupported cache dtype {cache.dtype}")


# ------------------------------------------------------------------ misc ---
def pa_abi_version() -> int:
    return int(lib().pa_abi_version())


def pa_get_device_error() -> int:
    v = ctypes.c_uint32(0)
    _check("pa_get_device_error", lib().pa_get_device_error(ctypes.byref(v)))
    return int(v.value)


# ----------------------------------------------------------------- cache ---
def pa_cache_write(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None):
    """Scatter k_new/v_new [T, Hkv, d] into the pools at slot_mapping[T]."""
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    nb, hkv, bs, d = k_cache.shape
    _need(k_new, k_cache.dtype, "k_new", 3)
    _need(v_new, k_cache.dtype, "v_new", 3)
    _check("pa_cache_write", lib().pa_cache_write(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), k_new.shape[0], _ptr(k_cache),
        _ptr(v_cache), nb, hkv, bs, d, _kv_dtype(k_cache), _stream(stream)))


def pa_cache_write_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                       stream=None):
    """Append bf16 k_new/v_new [T, Hkv, d] to an E4M3 cache (uint8 pools,
    fp32 scales [num_blocks, Hkv]) at slot_mapping[T]; grow-only scales."""
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(k_scale, torch.float32, "k_scale", 2)
    _need(v_scale, torch.float32, "v_scale", 2)
    if _kv_dtype(k_cache) != PA_KV_FP8_E4M3:
        raise TypeError("pa_cache_write_fp8: the cache must hold E4M3 bytes")
    nb, hkv, bs, d = k_cache.shape
    _check("pa_cache_write_fp8", lib().pa_cache_write_fp8(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), k_new.shape[0], _ptr(k_cache),
        _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), nb, hkv, bs, d, _stream(stream)))


def pa_swap_out(k_cache, v_cache, block_ids, host_k, host_v, k_scale=None, v_scale=None,
                host_k_scale=None, host_v_scale=None, stream=None):
    """Copy the listed blocks (device int32 ids) of the pools into pinned
    host tensors [n, Hkv, bs, d] (and FP8 scales [n, Hkv])."""
    _need(block_ids, torch.int32, "block_ids", 1)
    nb, hkv, bs, d = k_cache.shape
    _check("pa_swap_out", lib().pa_swap_out(
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_ids),
        block_ids.shape[0], _ptr(host_k), _ptr(host_v), _ptr(host_k_scale),
        _ptr(host_v_scale), nb, hkv, bs, d, _kv_dtype(k_cache), _stream(stream)))


def pa_swap_in(host_k, host_v, block_ids, k_cache, v_cache, host_k_scale=None,
               host_v_scale=None, k_scale=None, v_scale=None, stream=None):
    """The reverse of pa_swap_out: pinned host slots i -> blocks block_ids[i]."""
    _need(block_ids, torch.int32, "block_ids", 1)
    nb, hkv, bs, d = k_cache.shape
    _check("pa_swap_in", lib().pa_swap_in(
        _ptr(host_k), _ptr(host_v), _ptr(host_k_scale), _ptr(host_v_scale), _ptr(block_ids),
        block_ids.shape[0], _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), nb,
        hkv, bs, d, _kv_dtype(k_cache), _stream(stream)))


def pa_copy_blocks(k_cache, v_cache, pairs, k_scale=None, v_scale=None, stream=None):
    """Copy-on-write: pairs int32 [P, 3] rows (src, dst, valid slots)."""
    _need(pairs, torch.int32, "pairs", 2)
    nb, hkv, bs, d = k_cache.shape
    _check("pa_copy_blocks", lib().pa_copy_blocks(
        _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(pairs),
        pairs.shape[0], nb, hkv, bs, d, _kv_dtype(k_cache), _stream(stream)))


def pa_quantize_fp8(k_src, v_src, block_ids, valid_lens, k_dst, v_dst, k_scale,
                    v_scale, stream=None):
    """Quantise listed bf16 blocks to E4M3 with per-(block, head) scales."""
    _need(block_ids, torch.int32, "block_ids", 1)
    _need(valid_lens, torch.int32, "valid_lens", 1)
    _need(k_scale, torch.float32, "k_scale", 2)
    _need(v_scale, torch.float32, "v_scale", 2)
    nb, hkv, bs, d = k_src.shape
    _check("pa_quantize_fp8", lib().pa_quantize_fp8(
        _ptr(k_src), _ptr(v_src), _ptr(block_ids), _ptr(valid_lens), block_ids.shape[0],
        _ptr(k_dst), _ptr(v_dst), _ptr(k_scale), _ptr(v_scale), nb, hkv, bs, d,
        _stream(stream)))


# ---------------------------------------------------------------- decode ---
def pa_testing_set_wait_limit(polls: int, stall: bool = False):
    """Test hook (include/pa_testing.h): polls before a decode pipeline wait
    gives up (0 restores the default and clears stall); stall=True makes
    every decode CTA first wait on a barrier nothing arrives at."""
    _check("pa_testing_set_wait_limit", lib().pa_testing_set_wait_limit(polls, int(stall)))


def pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                             num_splits=0) -> int:
    n = ctypes.c_size_t(0)
    _check("pa_decode_workspace_size", lib().pa_decode_workspace_size(
        num_seqs, num_q_heads, num_kv_heads, head_dim, num_splits, ctypes.byref(n)))
    return int(n.value)


def pa_decode(q, k_cache, v_cache, block_tables, seq_lens, scale, out, workspace=None,
              k_scale=None, v_scale=None, num_splits=0, stream=None):
    """Paged decode attention: out[B, Hq, d] (bf16) from q[B, Hq, d] (bf16).
    ``seq_lens`` is read before the wait for the preceding kernel (see the
    module docstring)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_decode", lib().pa_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _kv_dtype(k_cache), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B,
        hq, hkv, d, bs, nb, float(scale), _ptr(out), _ptr(workspace), ws_bytes, num_splits,
        _stream(stream)))


def pa_decode_append(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, seq_lens,
                     scale, out, workspace=None, num_splits=0, stream=None):
    """This step's cache write and decode in one launch (bf16 cache): the
    same cache and out as pa_cache_write(k_new, v_new, slot_mapping, ...)
    then pa_decode(...), where row b of k_new / v_new is sequence b's new
    token and slot_mapping[b] its slot (< 0: none)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(out, torch.bfloat16, "out", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    if k_cache.dtype != torch.bfloat16 or v_cache.dtype != torch.bfloat16:
        raise ValueError("pa_decode_append: the cache must be bf16")
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if tuple(k_new.shape) != (B, hkv, d) or tuple(v_new.shape) != (B, hkv, d) or \
            slot_mapping.shape[0] != B:
        raise ValueError("pa_decode_append: k_new/v_new must be [B, Hkv, d], slot_mapping [B]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_decode_append", lib().pa_decode_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B, hq, hkv, d, bs, nb,
        float(scale), _ptr(out), _ptr(workspace), ws_bytes, num_splits, _stream(stream)))


def pa_decode_append_fp8(q, k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                         block_tables, seq_lens, scale, out, workspace=None, num_splits=0,
                         stream=None):
    """The FP8 decode step in one launch: pa_cache_write_fp8 of row b of
    k_new / v_new at slot_mapping[b], then pa_decode, bit for bit (block
    size 8 or 16)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(k_scale, torch.float32, "k_scale", 2)
    _need(v_scale, torch.float32, "v_scale", 2)
    _need(out, torch.bfloat16, "out", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    if _kv_dtype(k_cache) != PA_KV_FP8_E4M3:
        raise TypeError("pa_decode_append_fp8: the cache must hold E4M3 bytes")
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_decode_append_fp8", lib().pa_decode_append_fp8(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
        _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), B, hq, hkv, d, bs, nb, float(scale), _ptr(out), _ptr(workspace),
        ws_bytes, num_splits, _stream(stream)))


# ----------------------------------------------------------------- NVFP4 ---
def nvfp4_empty_cache(num_blocks, num_kv_heads, block_size, head_dim, device="cuda"):
    """Zeroed NVFP4 pools (k, k_sf, v, v_sf), uint8, in the layout of
    include/pa.h: k [nb, Hkv, bs, d/2], k_sf [nb, Hkv, bs, d/16],
    v [nb, Hkv, bs/2, d], v_sf [nb, Hkv, d/16, bs]."""
    nb, h, bs, d = num_blocks, num_kv_heads, block_size, head_dim
    z = lambda *shape: torch.zeros(shape, dtype=torch.uint8, device=device)
    return z(nb, h, bs, d // 2), z(nb, h, bs, d // 16), z(nb, h, bs // 2, d), z(nb, h, d // 16, bs)


def _nvfp4_dims(cache):
    k, k_sf, v, v_sf = cache
    for t, n in zip(cache, ("k", "k_sf", "v", "v_sf")):
        _need(t, torch.uint8, n, 4)
    nb, hkv, bs, d2 = k.shape
    d = 2 * d2
    if tuple(k_sf.shape) != (nb, hkv, bs, d // 16) or tuple(v.shape) != (nb, hkv, bs // 2, d) \
            or tuple(v_sf.shape) != (nb, hkv, d // 16, bs):
        raise ValueError("NVFP4 cache: inconsistent pool shapes")
    return nb, hkv, bs, d


def pa_cache_write_nvfp4(k_new, v_new, slot_mapping, cache, k_gscale, v_gscale, stream=None):
    """Quantise k_new/v_new [T, Hkv, d] (bf16) into the NVFP4 pools
    cache = (k, k_sf, v, v_sf) at slot_mapping[T] with tensor scales
    k_gscale / v_gscale."""
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    nb, hkv, bs, d = _nvfp4_dims(cache)
    k, k_sf, v, v_sf = cache
    _check("pa_cache_write_nvfp4", lib().pa_cache_write_nvfp4(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), k_new.shape[0], _ptr(k), _ptr(v),
        _ptr(k_sf), _ptr(v_sf), float(k_gscale), float(v_gscale), nb, hkv, bs, d,
        _stream(stream)))


def pa_decode_nvfp4(q, cache, k_gscale, v_gscale, block_tables, seq_lens, scale, out,
                    workspace=None, num_splits=0, stream=None):
    """Paged decode attention over NVFP4 pools cache = (k, k_sf, v, v_sf)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    nb, hkv, bs, d = _nvfp4_dims(cache)
    k, k_sf, v, v_sf = cache
    B, hq, dq = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_decode_nvfp4", lib().pa_decode_nvfp4(
        _ptr(q), _ptr(k), _ptr(v), _ptr(k_sf), _ptr(v_sf), float(k_gscale), float(v_gscale),
        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B, hq, hkv, dq, bs, nb,
        float(scale), _ptr(out), _ptr(workspace), ws_bytes, num_splits, _stream(stream)))


def pa_decode_append_nvfp4(q, k_new, v_new, slot_mapping, cache, k_gscale, v_gscale,
                           block_tables, seq_lens, scale, out, workspace=None, num_splits=0,
                           stream=None):
    """The NVFP4 decode step in one launch: pa_cache_write_nvfp4 of row b of
    k_new / v_new at slot_mapping[b], then pa_decode_nvfp4, bit for bit."""
    _need(q, torch.bfloat16, "q", 3)
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(out, torch.bfloat16, "out", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    nb, hkv, bs, d = _nvfp4_dims(cache)
    k, k_sf, v, v_sf = cache
    B, hq, dq = q.shape
    if tuple(k_new.shape) != (B, hkv, dq) or tuple(v_new.shape) != (B, hkv, dq) or \
            slot_mapping.shape[0] != B:
        raise ValueError("pa_decode_append_nvfp4: k_new/v_new must be [B, Hkv, d], "
                         "slot_mapping [B]")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_decode_append_nvfp4", lib().pa_decode_append_nvfp4(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k), _ptr(v), _ptr(k_sf),
        _ptr(v_sf), float(k_gscale), float(v_gscale), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), B, hq, hkv, dq, bs, nb, float(scale), _ptr(out), _ptr(workspace),
        ws_bytes, num_splits, _stream(stream)))


def pa_decode_cascade_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                     block_size, prefix_len, num_splits=0):
    n = _c_size(0)
    _check("pa_decode_cascade_workspace_size", lib().pa_decode_cascade_workspace_size(
        num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, prefix_len, num_splits,
        ctypes.byref(n)))
    return n.value


def pa_decode_cascade(q, k_cache, v_cache, block_tables, seq_lens, prefix_len, scale, out,
                      workspace, num_splits=0, stream=None):
    """pa_decode for a batch whose sequences share their first prefix_len
    tokens (the same physical blocks): the prefix is read once."""
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    if k_cache.dtype != torch.bfloat16 or v_cache.dtype != torch.bfloat16:
        raise ValueError("pa_decode_cascade: the cache must be bf16")
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("pa_decode_cascade", lib().pa_decode_cascade(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), B, hq, hkv, d, bs, nb, int(prefix_len), float(scale), _ptr(out),
        _ptr(workspace), ws_bytes, num_splits, _stream(stream)))


NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def pa_decode_noalloc(q, k_cache, v_cache, block_tables, seq_lens, scale, out,
                      k_scale=None, v_scale=None, num_splits=0, stream=None):
    """pa_decode without a workspace argument, for callers that cannot
    allocate device memory: the library's own 16 MiB device array serves as
    scratch.  Calls on one device share it, so calls whose kernels overlap
    (unordered streams) race; requests needing more scratch raise
    PA_ERR_WORKSPACE."""
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    _check("pa_decode_noalloc", lib().pa_decode_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _kv_dtype(k_cache), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B,
        hq, hkv, d, bs, nb, float(scale), _ptr(out), num_splits, _stream(stream)))


# --------------------------------------------------------- block manager ---
class Allocator:
    """Handle over the native host block manager (pa_allocator)."""

    def __init__(self, num_blocks: int):
        h = ctypes.c_void_p()
        _check("pa_allocator_create", lib().pa_allocator_create(num_blocks, ctypes.byref(h)))
        self._h = h
        self.num_blocks = num_blocks

    def close(self):
        if self._h:
            lib().pa_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _ids(ids):
        arr = (ctypes.c_int32 * max(1, len(ids)))(*ids)
        return arr, len(ids)

    def alloc(self, n: int):
        """(status, ids or None)."""
        buf = (ctypes.c_int32 * max(1, n))()
        st = lib().pa_block_alloc(self._h, n, buf)
        return st, (list(buf[:n]) if st == PA_OK else None)

    def free(self, ids) -> int:
        arr, n = self._ids(ids)
        return lib().pa_block_free(self._h, arr, n)

    def fork(self, ids) -> int:
        arr, n = self._ids(ids)
        return lib().pa_block_fork(self._h, arr, n)

    def refcount(self, bid: int):
        rc = ctypes.c_int32(0)
        st = lib().pa_block_refcount(self._h, bid, ctypes.byref(rc))
        return st, (rc.value if st == PA_OK else None)

    def num_free(self) -> int:
        return int(lib().pa_block_num_free(self._h))

    def append_slots(self, table: list, length: int, n: int, block_size: int,
                     max_blocks: int):
        """Grow a sequence; ``table`` (list) is updated in place on success.

        Returns (status, slots, cow_pairs) like the C call.
        """
        tab = (ctypes.c_int32 * max(1, max_blocks))(*([-1] * max(1, max_blocks)))
        for i, b in enumerate(table[:max_blocks]):
            tab[i] = b
        slots = (ctypes.c_int64 * max(1, n))()
        cow = (ctypes.c_int32 * 3)()
        ncow = ctypes.c_int32(0)
        st = lib().pa_seq_append_slots(self._h, tab, max_blocks, length, n, block_size,
                                       slots, cow, ctypes.byref(ncow))
        if st != PA_OK:
            return st, None, None
        # the call filled the -1 padded table up to the sequence's new end
        table[:] = list(itertools.takewhile(lambda x: x >= 0, tab))
        pairs = [tuple(cow[:3])] if ncow.value else []
        return st, list(slots[:n]), pairs


class BatchAppender:
    """One decode step's appends for a batch through pa_batch_append_slots.

    Holds host arrays sized for the batch so that each call is one native
    call with no per-sequence Python work: ``tables`` (int32 [B, max_blocks],
    -1 padded) is updated in place.
    """

    def __init__(self, alloc: "Allocator", tables, max_blocks: int):
        import numpy as np
        self.alloc = alloc
        self.max_blocks = max_blocks
        B = len(tables)
        self.tables = np.full((B, max_blocks), -1, dtype=np.int32)
        for b, t in enumerate(tables):
            self.tables[b, :len(t)] = t
        self.cow = np.zeros((B, 3), dtype=np.int32)
        self.ncow = np.zeros(B, dtype=np.int32)

    def append(self, lens, n_new, block_size: int):
        """(status, slots int64 [sum n_new], cow pairs list, num_done)."""
        import numpy as np
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        n_new = np.ascontiguousarray(n_new, dtype=np.int32)
        slots = np.zeros(max(1, int(n_new.sum())), dtype=np.int64)
        done = ctypes.c_int32(0)
        fn = lib().pa_batch_append_slots
        args = (self.alloc._h, self.tables.ctypes.data, self.max_blocks, lens.ctypes.data,
                n_new.ctypes.data, len(lens), block_size, slots.ctypes.data,
                self.cow.ctypes.data, self.ncow.ctypes.data, ctypes.byref(done))
        t0 = time.perf_counter()
        st = fn(*args)
        self.last_call_us = (time.perf_counter() - t0) * 1e6  # the native call alone
        pairs = [tuple(int(x) for x in self.cow[i]) for i in np.flatnonzero(self.ncow[:done.value])]
        return st, slots[:int(n_new[:done.value].sum())], pairs, done.value


def allocator_usage(alloc: "Allocator", tables, lens, block_size: int) -> dict:
    """pa_allocator_usage over the sequences (tables: lists or an int32
    [B, max_blocks] array; lens: per-sequence lengths)."""
    import numpy as np
    if isinstance(tables, np.ndarray):
        tab = np.ascontiguousarray(tables, dtype=np.int32)
    else:
        width = max([1] + [len(t) for t in tables])
        tab = np.full((len(tables), width), -1, dtype=np.int32)
        for b, t in enumerate(tables):
            tab[b, :len(t)] = t
    ln = np.ascontiguousarray(lens, dtype=np.int32)
    out = np.zeros(4, dtype=np.int64)
    _check("pa_allocator_usage", lib().pa_allocator_usage(
        alloc._h, tab.ctypes.data, tab.shape[1], ln.ctypes.data, len(ln), block_size,
        out.ctypes.data))
    return dict(zip(("live_blocks", "slots_reserved", "tokens_stored", "tokens_logical"),
                    (int(x) for x in out)))


def replay_script(ops, num_seqs: int, block_size: int, max_blocks: int, num_blocks: int):
    """Apply a workload op script to a fresh native allocator.

    Returns (allocator, tables, lens); raises on any non-OK status.
    """
    a = Allocator(num_blocks)
    tables = [[] for _ in range(num_seqs)]
    lens = [0] * num_seqs
    for op in ops:
        kind = op[0]
        if kind == "alloc":
            st, _ = a.alloc(op[1])
            _check("pa_block_alloc", st)
        elif kind == "free_list":
            _check("pa_block_free", a.free(op[1]))
        elif kind == "append":
            _, b, n = op
            st, _, _ = a.append_slots(tables[b], lens[b], n, block_size, max_blocks)
            _check("pa_seq_append_slots", st)
            lens[b] += n
        elif kind == "fork":
            _, child, parent, ntok = op
            ids = tables[parent][:-(-ntok // block_size)]
            _check("pa_block_fork", a.fork(ids))
            tables[child] = list(ids)
            lens[child] = ntok
        else:
            raise ValueError(kind)
    return a, tables, lens
