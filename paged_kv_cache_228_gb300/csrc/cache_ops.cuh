// Cache maintenance kernels: scatter append, copy-on-write block copy and
// per-(block, head) FP8 quantisation.  All are bandwidth-trivial next to the
// decode step (they touch only the new tokens, the copied blocks or the
// quantised blocks) and are written as plain 16-byte vectorised copies.
#pragma once

#include "pa_device.cuh"

namespace pa {

// --------------------------------------------------------- cache write ---
// "Paged Attention and KV Cache Fragmentation", section "How PagedAttention
// maps an OS concept onto GPU memory": each new token's K/V goes to the
// slot its block table names.  One thread per 16-byte chunk; consecutive
// threads cover one (token, head) row, K rows then V rows.
__global__ void __launch_bounds__(256)
    cache_write_kernel(const uint4* __restrict__ k_new,
                       const uint4* __restrict__ v_new,
                       const int64_t* __restrict__ slots, int32_t num_tokens,
                       uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       int64_t num_slots, int32_t num_kv_heads,
                       int32_t block_size, int32_t chunks_per_row) {
  // Launched as a programmatic dependent: wait for the previous grid
  // before reading any input, then let the next grid begin launching.
  pdl_wait();
  pdl_trigger();
  const int64_t per_token = 2LL * num_kv_heads * chunks_per_row;
  const int64_t total = per_token * num_tokens;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       i < total; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / per_token;
    int64_t r = i - t * per_token;
    const int kv = static_cast<int>(r / (static_cast<int64_t>(num_kv_heads) * chunks_per_row));
    r -= static_cast<int64_t>(kv) * num_kv_heads * chunks_per_row;
    const int32_t h = static_cast<int32_t>(r / chunks_per_row);
    const int32_t c = static_cast<int32_t>(r - static_cast<int64_t>(h) * chunks_per_row);
    const int64_t s = slots[t];
    if (s < 0) continue;
    if (s >= num_slots) {
      if (kv == 0 && h == 0 && c == 0) flag_error(PA_DEVERR_BAD_SLOT);
      continue;
    }
    const int64_t blk = s / block_size, off = s - blk * block_size;
    const int64_t src = (t * num_kv_heads + h) * chunks_per_row + c;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * chunks_per_row + c;
    if (kv == 0)
      k_cache[dst] = k_new[src];
    else
      v_cache[dst] = v_new[src];
  }
}

// ---------------------------------------------------------- block copy ---
// Copy-on-write of a shared partial block (same page, the shared-prefix
// paragraph): grid (pairs, heads, K/V); each CTA copies the first n rows of
// one head of one block.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       float* __restrict__ k_scale, float* __restrict__ v_scale,
                       const int32_t* __restrict__ pairs, int32_t num_blocks,
                       int32_t num_kv_heads, int32_t block_size,
                       int32_t chunks_per_row) {
  const int32_t pr = blockIdx.x, h = blockIdx.y, kv = blockIdx.z;
  const int32_t src = pairs[3 * pr], dst = pairs[3 * pr + 1], n = pairs[3 * pr + 2];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks || n < 0 ||
      n > block_size) {
    if (threadIdx.x == 0 && h == 0 && kv == 0) flag_error(PA_DEVERR_BAD_PAIR);
    return;
  }
  uint4* cache = kv == 0 ? k_cache : v_cache;
  const int64_t row = static_cast<int64_t>(block_size) * chunks_per_row;
  const uint4* s = cache + (static_cast<int64_t>(src) * num_kv_heads + h) * row;
  uint4* d = cache + (static_cast<int64_t>(dst) * num_kv_heads + h) * row;
  const int32_t cnt = n * chunks_per_row;
  for (int32_t i = threadIdx.x; i < cnt; i += blockDim.x) d[i] = s[i];
  float* sc = kv == 0 ? k_scale : v_scale;
  if (sc != nullptr && threadIdx.x == 0)
    sc[static_cast<int64_t>(dst) * num_kv_heads + h] =
        sc[static_cast<int64_t>(src) * num_kv_heads + h];
}

// ------------------------------------------------------- FP8 quantise ---
// "Paged Attention and KV Cache Fragmentation", section "Quantization as a
// way to stretch paged memory further".  One CTA per (listed block, head,
// K/V): absmax over the valid rows, scale = absmax / 448 (IEEE division),
// codes = e4m3_rne_satfinite(x / scale) (IEEE division per element), rows
// past the valid length written as +0.
__global__ void __launch_bounds__(256)
    quantize_fp8_kernel(const uint4* __restrict__ k_src,
                        const uint4* __restrict__ v_src,
                        const int32_t* __restrict__ block_ids,
                        const int32_t* __restrict__ valid_lens,
                        uint2* __restrict__ k_dst, uint2* __restrict__ v_dst,
                        float* __restrict__ k_scale, float* __restrict__ v_scale,
                        int32_t num_blocks, int32_t num_kv_heads,
                        int32_t block_size, int32_t head_dim) {
  const int32_t i = blockIdx.x, h = blockIdx.y, kv = blockIdx.z;
  const int32_t blk = block_ids[i], n = valid_lens[i];
  if (blk < 0 || blk >= num_blocks || n < 0 || n > block_size) {
    if (threadIdx.x == 0 && h == 0 && kv == 0) flag_error(PA_DEVERR_BAD_BLOCK_ID);
    return;
  }
  const int32_t vec_per_row = head_dim / 8;  // 8 elements per 16 bytes
  const int64_t tile = (static_cast<int64_t>(blk) * num_kv_heads + h) *
                       static_cast<int64_t>(block_size) * vec_per_row;
  const uint4* src = (kv == 0 ? k_src : v_src) + tile;
  uint2* dst = (kv == 0 ? k_dst : v_dst) + tile;
  const int32_t nvec = block_size * vec_per_row;
  const int32_t nvalid = n * vec_per_row;

  float amax = 0.f;
  for (int32_t j = threadIdx.x; j < nvalid; j += blockDim.x) {
    const uint4 w = src[j];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = unpack_bf16x2(ws[q]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float red[8];
  __shared__ float s_scale;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) a = fmaxf(a, red[w]);
    const float scale = a == 0.f ? 1.f : __fdiv_rn(a, 448.f);
    s_scale = scale;
    (kv == 0 ? k_scale : v_scale)[static_cast<int64_t>(blk) * num_kv_heads + h] = scale;
  }
  __syncthreads();
  const float scale = s_scale;
  for (int32_t j = threadIdx.x; j < nvec; j += blockDim.x) {
    uint2 out = make_uint2(0u, 0u);
    if (j < nvalid) {
      const uint4 w = src[j];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      uint32_t codes[2] = {0u, 0u};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = unpack_bf16x2(ws[q]);
        const uint32_t c0 = __nv_cvt_float_to_fp8(__fdiv_rn(f.x, scale), __NV_SATFINITE, __NV_E4M3);
        const uint32_t c1 = __nv_cvt_float_to_fp8(__fdiv_rn(f.y, scale), __NV_SATFINITE, __NV_E4M3);
        codes[q >> 1] |= (c0 | (c1 << 8)) << ((q & 1) * 16);
      }
      out = make_uint2(codes[0], codes[1]);
    }
    dst[j] = out;
  }
}

// FP8 append ("Paged Attention and KV Cache Fragmentation", section
// "Quantization as a way to stretch paged memory further", for the FP8
// cache; appending into a partly filled block is this library's reading).
// One warp per (token t, KV head h, K|V); lane l owns bytes
// [l * D/32, (l+1) * D/32) of every row.  With s_t = absmax(x) / 448:
//   offset 0:        scale = s_t (1 when the row is all zero)
//   s_t > old scale: scale = s_t, and earlier rows r < offset become
//                    e4m3(fp32(decode(code) * old) / scale)
//   otherwise:       the scale stays
// then the row is e4m3(x / scale) (fp32 IEEE division, RNE, satfinite).
// Tokens of one call must name distinct blocks (a block updated by two
// warps at once ends unspecified).  With `tables` non-null, token t is
// sequence t's appended token of a decode step: a slot other than the one
// the table gives position seq_lens[t] - 1 (or any slot of an empty
// sequence) is not written and flags PA_DEVERR_BAD_SLOT.
template <int D>
__global__ void __launch_bounds__(256, 1)
    cache_write_fp8_kernel(const __nv_bfloat16* __restrict__ k_new,
                           const __nv_bfloat16* __restrict__ v_new,
                           const int64_t* __restrict__ slots, int32_t num_tokens,
                           uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                           float* __restrict__ k_scale, float* __restrict__ v_scale,
                           int64_t num_slots, int32_t num_kv_heads, int32_t block_size,
                           const int32_t* __restrict__ seq_lens,
                           const int32_t* __restrict__ tables, int32_t max_blocks) {
  pdl_wait();  // as cache_write_kernel
  pdl_trigger();
  constexpr int E = D / 32;  // bytes (and elements) per lane per row
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (wid >= static_cast<int64_t>(num_tokens) * num_kv_heads * 2) return;
  const int kv = static_cast<int>(wid & 1);
  const int64_t th = wid >> 1;
  const int32_t h = static_cast<int32_t>(th % num_kv_heads);
  const int64_t t = th / num_kv_heads;
  const int64_t s = slots[t];
  if (s < 0) return;
  if (s >= num_slots) {
    if (lane == 0 && h == 0 && kv == 0) flag_error(PA_DEVERR_BAD_SLOT);
    return;
  }
  if (tables != nullptr) {
    const int32_t n = seq_lens[t];
    bool at_end = n > 0 && static_cast<int64_t>(n) <= static_cast<int64_t>(max_blocks) * block_size;
    if (at_end) {
      const int32_t pos = n - 1;
      at_end = static_cast<int64_t>(tables[t * max_blocks + pos / block_size]) * block_size +
                   pos % block_size == s;
    }
    if (!at_end) {
      if (lane == 0 && h == 0 && kv == 0) flag_error(PA_DEVERR_BAD_SLOT);
      return;
    }
  }
  const int64_t blk = s / block_size;
  const int32_t off = static_cast<int32_t>(s - blk * block_size);

  const __nv_bfloat16* src = (kv ? v_new : k_new) + (t * num_kv_heads + h) * D + lane * E;
  float x[E];
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const float2 f = unpack_bf16x2(*reinterpret_cast<const uint32_t*>(src + i));
    x[i] = f.x;
    x[i + 1] = f.y;
    a = fmaxf(a, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));

  float* sp = (kv ? v_scale : k_scale) + blk * num_kv_heads + h;
  uint8_t* rows = (kv ? v_cache : k_cache) + (blk * num_kv_heads + h) * block_size * D + lane * E;
  const float old = *sp;
  const float st = __fdiv_rn(a, 448.f);
  float sc = old;
  if (off == 0) {
    sc = a == 0.f ? 1.f : st;
  } else if (st > old) {
    sc = st;
    for (int32_t r = 0; r < off; ++r) {
      uint8_t* row = rows + static_cast<int64_t>(r) * D;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const __half_raw hr = __nv_cvt_fp8_to_halfraw(row[i], __NV_E4M3);
        const float y = __fmul_rn(__half2float(__half(hr)), old);
        row[i] = __nv_cvt_float_to_fp8(__fdiv_rn(y, sc), __NV_SATFINITE, __NV_E4M3);
      }
    }
  }
  uint8_t* row = rows + static_cast<int64_t>(off) * D;
#pragma unroll
  for (int i = 0; i < E; ++i)
    row[i] = __nv_cvt_float_to_fp8(__fdiv_rn(x[i], sc), __NV_SATFINITE, __NV_E4M3);
  if (lane == 0) *sp = sc;
}

// Block swap between the device pools and host memory the GPU addresses
// directly ("Paged Attention and KV Cache Fragmentation", section
// "Offloading paged KV blocks to CPU DRAM and NVMe": blocks move down to
// host memory for headroom and back).  On
// a GB300 the host side sits behind NVLink-C2C, so the kernel reads or
// writes it in place (zero-copy) instead of issuing a copy per block.
// Listed block i <-> host slot i ([num_ids][Hkv][bs][row bytes] for K and
// for V, and [num_ids][Hkv] FP8 scales).  16-byte chunks, grid-stride, four
// in flight per thread.
__global__ void __launch_bounds__(256)
    swap_blocks_kernel(uint4* __restrict__ dev_k, uint4* __restrict__ dev_v,
                       float* __restrict__ dev_ks, float* __restrict__ dev_vs,
                       uint4* __restrict__ host_k, uint4* __restrict__ host_v,
                       float* __restrict__ host_ks, float* __restrict__ host_vs,
                       const int32_t* __restrict__ block_ids, int32_t num_ids,
                       int32_t num_blocks, int32_t num_kv_heads, int64_t block_chunks,
                       bool to_host) {
  pdl_wait();
  pdl_trigger();
  const int64_t per_id = 2 * block_chunks;  // K and V chunks of one block
  const int64_t total = per_id * num_ids;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < total;
       base += 4 * stride) {
    uint4 v[4];
    int64_t dst[4];
    bool ok[4];
    int kv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = base + u * stride;
      ok[u] = false;
      if (i >= total) continue;
      const int64_t id = i / per_id;
      const int64_t r = i - id * per_id;
      kv[u] = r >= block_chunks;
      const int64_t c = kv[u] ? r - block_chunks : r;
      const int32_t blk = block_ids[id];
      if (blk < 0 || blk >= num_blocks) {
        if (r == 0) flag_error(PA_DEVERR_BAD_BLOCK_ID);
        continue;
      }
      const int64_t dev = static_cast<int64_t>(blk) * block_chunks + c;
      const int64_t host = id * block_chunks + c;
      ok[u] = true;
      if (to_host) {
        v[u] = (kv[u] ? dev_v : dev_k)[dev];
        dst[u] = host;
      } else {
        v[u] = (kv[u] ? host_v : host_k)[host];
        dst[u] = dev;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (!ok[u]) continue;
      if (to_host)
        (kv[u] ? host_v : host_k)[dst[u]] = v[u];
      else
        (kv[u] ? dev_v : dev_k)[dst[u]] = v[u];
    }
  }
  // FP8 scales: one float per (block, head), K and V
  if (dev_ks != nullptr) {
    const int64_t ns = static_cast<int64_t>(num_ids) * num_kv_heads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < ns;
         i += stride) {
      const int64_t id = i / num_kv_heads, h = i - id * num_kv_heads;
      const int32_t blk = block_ids[id];
      if (blk < 0 || blk >= num_blocks) continue;
      const int64_t d = static_cast<int64_t>(blk) * num_kv_heads + h;
      if (to_host) {
        host_ks[i] = dev_ks[d];
        host_vs[i] = dev_vs[d];
      } else {
        dev_ks[d] = host_ks[i];
        dev_vs[d] = host_vs[i];
      }
    }
  }
}

}  // namespace pa
