// Shared-prefix pass of the cascade decode.
//
// "Paged Attention and KV Cache Fragmentation", section "How PagedAttention
// maps an OS concept onto GPU memory", and the "KV cache fragmentation"
// field guide, section "Why it matters": sequences forked from one prompt
// point at the same physical prefix blocks.  Attention over a sequence is
// the log-sum-exp merge of attention over any split of its tokens, so the
// prefix part can be computed once for every sequence's queries: for KV
// head g it is a dense product of all B*G query rows with the prefix keys
// and values, S = Q_g K_p^T, online softmax, O = P V_p -- a contraction
// with many rows, run here on the tensor pipe (mma.sync m16n8k16, queries
// on M, tokens on N for QK and on K for PV).  The result is one partial
// (o unnormalised, m in log2 units, l) per (sequence, query head); the
// suffix decode and its merge fold it in.
//
// CTA = 4 warps on 64 query rows of one KV head and one of S token ranges
// of the prefix (S splits keep ~3 CTAs per SM busy).  The CTA streams its
// range in 32-token chunks through a 3-stage cp.async ring that all 4
// warps read (each chunk's K and V are fetched once per 64 rows); warp w
// computes rows 16w .. 16w+15.  Chunk rows use the decode kernels' 128-byte
// slab layout with the chunk index XOR-swizzled by row, and the range's
// block ids are staged in shared memory first.  Each split writes its own
// partial; the consumers fold in all S.
#pragma once

#include "pa_device.cuh"

namespace pa {

struct PrefixParams {
  const uint8_t* q;        // [num_seqs][num_q_heads][D] bf16
  const uint8_t* k_cache;  // [num_blocks][num_kv_heads][block_size][D] bf16
  const uint8_t* v_cache;
  const int32_t* prefix_table;  // the prefix's block ids (sequence 0's table)
  float* pf_o;                  // [splits][num_seqs * num_q_heads][D]
  float2* pf_ml;                // [splits][num_seqs * num_q_heads]
  int32_t num_seqs, num_q_heads, num_kv_heads, group, block_size, log2_bs, num_blocks;
  int32_t prefix_tokens;
  int32_t prefix_chunks;  // ceil(prefix_tokens / 32)
  int32_t splits;         // S
  float scale_log2;
};

constexpr int kPfWarps = 4;
constexpr int kPfRows = 64;     // query rows per CTA (16 per warp)
constexpr int kPfChunk = 32;    // tokens per stage
constexpr int kPfStages = 3;
constexpr int kPfMaxBlocks = 1024;  // block ids of one split staged in shared memory

template <int D>
struct PfSmem {
  static constexpr int kRows128 = 128;                   // bytes per slab row
  static constexpr int kKV = (D / 64) * kPfChunk * 128;  // K (or V) of a chunk
  static constexpr int kStage = 2 * kKV;
  static constexpr int kQ = (D / 64) * kPfRows * 128;
  static constexpr int kIds = kPfMaxBlocks * 4;
  static constexpr int kBytes = kQ + kPfStages * kStage + kIds;
};

// Byte offset of 16-byte chunk c (along the row's D * 2 bytes) of row r in
// a tile of `rows` rows stored as 128-byte slabs.
__device__ __forceinline__ uint32_t pf_chunk(int rows, int r, int c) {
  return (c >> 3) * (rows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most n (0..2) of this thread's copy groups are in flight.
__device__ __forceinline__ void cp_async_wait_upto(int n) {
  if (n >= 2)
    asm volatile("cp.async.wait_group 2;" ::: "memory");
  else if (n == 1)
    asm volatile("cp.async.wait_group 1;" ::: "memory");
  else
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// CTA: K and V rows of prefix chunk ch (its block ids in `ids`, indexed
// from the split's first block) into a stage.  Invalid ids read as zeros.
template <int D>
__device__ __forceinline__ void pf_issue(const PrefixParams& p, int32_t g, int32_t ch,
                                         int32_t first_tok, const int32_t* ids,
                                         uint32_t kdst) {
  constexpr int kCpr = D * 2 / 16;  // chunks per row
  for (int idx = threadIdx.x; idx < kPfChunk * kCpr; idx += kPfWarps * 32) {
    const int r = idx / kCpr, c = idx % kCpr;
    const int32_t tok = ch * kPfChunk + r;
    // rows past the prefix (a last chunk of 16) read as zeros
    const int32_t blk = tok < p.prefix_tokens ? ids[(tok - first_tok) >> p.log2_bs] : -1;
    const bool ok = blk >= 0 && blk < p.num_blocks;
    const int64_t row = (static_cast<int64_t>(blk) * p.num_kv_heads + g) * p.block_size +
                        (tok & (p.block_size - 1));
    const int64_t byte = ok ? row * (D * 2) + c * 16 : 0;
    const uint32_t d = kdst + pf_chunk(kPfChunk, r, c);
    cp_async16(d, p.k_cache + byte, ok ? 16u : 0u);
    cp_async16(d + PfSmem<D>::kKV, p.v_cache + byte, ok ? 16u : 0u);
  }
}

template <int D>
__global__ void __launch_bounds__(kPfWarps * 32)
    prefix_attention_kernel(const PrefixParams p) {
  using L = PfSmem<D>;
  extern __shared__ __align__(1024) uint8_t pf_smem[];
  pdl_wait();  // launched as a programmatic dependent: inputs ready below
  pdl_trigger();
  const uint32_t base = smem_addr(pf_smem);
  const uint32_t qs = base, ring = base + L::kQ;
  int32_t* ids = reinterpret_cast<int32_t*>(pf_smem + L::kQ + kPfStages * L::kStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int32_t g = blockIdx.y, split = blockIdx.z;
  const int64_t R = static_cast<int64_t>(p.num_seqs) * p.group;  // query rows of head g
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kPfRows;
  // this split's chunks [c0, c1) and their block ids
  const int32_t c0 = static_cast<int32_t>(static_cast<int64_t>(p.prefix_chunks) * split / p.splits);
  const int32_t c1 = static_cast<int32_t>(static_cast<int64_t>(p.prefix_chunks) * (split + 1) / p.splits);
  const int32_t first_tok = c0 * kPfChunk;
  const int32_t first_blk = first_tok >> p.log2_bs;
  const int32_t last_tok = min(c1 * kPfChunk, p.prefix_tokens) - 1;
  const int32_t nblk = ((last_tok >> p.log2_bs) - first_blk) + 1;
  for (int i = threadIdx.x; i < nblk; i += blockDim.x) {
    const int32_t e = p.prefix_table[first_blk + i];
    if (!(e >= 0 && e < p.num_blocks)) flag_error(PA_DEVERR_BAD_BLOCK_ID);
    ids[i] = e;
  }
  // first_tok is block-aligned only when bs <= 32; index ids from the
  // split's first block
  const int32_t id_tok0 = first_blk << p.log2_bs;
  // ---- 64 query rows (zeros past R): row r -> sequence (row0+r) / G, head g*G + (row0+r) % G
  {
    constexpr int kCpr = D * 2 / 16;
    for (int idx = threadIdx.x; idx < kPfRows * kCpr; idx += blockDim.x) {
      const int r = idx / kCpr, c = idx % kCpr;
      const int64_t gr = row0 + r;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (gr < R) {
        const int64_t b = gr / p.group, j = gr % p.group;
        v = *reinterpret_cast<const uint4*>(
            p.q + ((b * p.num_q_heads + g * p.group + j) * D) * 2 + c * 16);
      }
      asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(qs + pf_chunk(kPfRows, r, c)),
                   "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                   : "memory");
    }
  }
  __syncthreads();  // ids and Q staged
  // prologue: the first two chunks
  const int32_t n = c1 - c0;
  for (int k = 0; k < 2 && k < n; ++k) {
    pf_issue<D>(p, g, c0 + k, id_tok0, ids, ring + k * L::kStage);
    cp_async_commit();
  }
  // A fragments of this warp's 16 rows of Q
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int i = lane >> 3;  // matrices (rows 0-7 | 8-15) x (k lo | k hi)
    const int r = 16 * warp + (lane & 7) + 8 * (i & 1);
    ldsm_x4(qs + pf_chunk(kPfRows, r, 2 * ks + (i >> 1)), qa[ks][0], qa[ks][1], qa[ks][2],
            qa[ks][3]);
  }
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};  // rows gq, gq + 8
  for (int32_t k = 0; k < n; ++k) {
    if (k + 2 < n) {
      pf_issue<D>(p, g, c0 + k + 2, id_tok0, ids, ring + ((k + 2) % kPfStages) * L::kStage);
      cp_async_commit();
    }
    cp_async_wait_upto(min(2, n - 1 - k));
    __syncthreads();  // chunk k landed for every thread's copies
    const uint32_t kb = ring + (k % kPfStages) * L::kStage;
    // S = Q K^T, 4 blocks of 8 tokens
    float s[4][4] = {};
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
      for (int nbp = 0; nbp < 2; ++nbp) {
        const int i = lane >> 3;  // (tokens +0-7 | +8-15) x (k lo | k hi)
        const int r = 16 * nbp + (lane & 7) + 8 * (i >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + pf_chunk(kPfChunk, r, 2 * ks + (i & 1)), b0, b1, b2, b3);
        mma_bf16(s[2 * nbp], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma_bf16(s[2 * nbp + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
    // online softmax in log2 units; the running max moves (and O is
    // rescaled) only when a score exceeds it by more than 8
    const int32_t tok0 = (c0 + k) * kPfChunk;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        s[nb][q] = tok0 + 8 * nb + 2 * tq + (q & 1) < p.prefix_tokens ? s[nb][q] * p.scale_log2
                                                                        : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[nb][0], s[nb][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nb][2], s[nb][3]));
    }
    if (__any_sync(0xffffffffu, mx0 > m[0] + 8.f || mx1 > m[1] + 8.f)) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float n0 = fmaxf(m[0], mx0), n1 = fmaxf(m[1], mx1);
      const float a0 = fast_exp2(m[0] - n0), a1 = fast_exp2(m[1] - n1);
      m[0] = n0;
      m[1] = n1;
      l[0] *= a0;
      l[1] *= a1;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][0] *= a0;
        o[i][1] *= a0;
        o[i][2] *= a1;
        o[i][3] *= a1;
      }
    }
    // O += P V over the chunk's two 16-token halves; P rounded to bf16 as
    // the A operand, and l sums the same rounded values
    const uint32_t vb = kb + L::kKV;
#pragma unroll
    for (int kt = 0; kt < 2; ++kt) {
      const uint32_t pa0 = pack_bf16x2(fast_exp2(s[2 * kt][0] - m[0]), fast_exp2(s[2 * kt][1] - m[0]));
      const uint32_t pa1 = pack_bf16x2(fast_exp2(s[2 * kt][2] - m[1]), fast_exp2(s[2 * kt][3] - m[1]));
      const uint32_t pa2 = pack_bf16x2(fast_exp2(s[2 * kt + 1][0] - m[0]), fast_exp2(s[2 * kt + 1][1] - m[0]));
      const uint32_t pa3 = pack_bf16x2(fast_exp2(s[2 * kt + 1][2] - m[1]), fast_exp2(s[2 * kt + 1][3] - m[1]));
      {
        const float2 f0 = unpack_bf16x2(pa0), f1 = unpack_bf16x2(pa1);
        const float2 f2 = unpack_bf16x2(pa2), f3 = unpack_bf16x2(pa3);
        l[0] += (f0.x + f0.y) + (f2.x + f2.y);
        l[1] += (f1.x + f1.y) + (f3.x + f3.y);
      }
#pragma unroll
      for (int pp = 0; pp < D / 16; ++pp) {
        const int i = lane >> 3;  // (tokens 0-7 | 8-15) x (d block 2pp | 2pp+1)
        const int r = 16 * kt + (lane & 7) + 8 * (i & 1);
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(vb + pf_chunk(kPfChunk, r, 2 * pp + (i >> 1)), v0, v1, v2, v3);
        mma_bf16(o[2 * pp], pa0, pa1, pa2, pa3, v0, v1);
        mma_bf16(o[2 * pp + 1], pa0, pa1, pa2, pa3, v2, v3);
      }
    }
    __syncthreads();  // every warp is done with the stage before it is refilled
  }
  l[0] += __shfl_xor_sync(0xffffffffu, l[0], 1);
  l[0] += __shfl_xor_sync(0xffffffffu, l[0], 2);
  l[1] += __shfl_xor_sync(0xffffffffu, l[1], 1);
  l[1] += __shfl_xor_sync(0xffffffffu, l[1], 2);
  // ---- this split's partial of rows gq and gq + 8 of the warp
  const int64_t stride = static_cast<int64_t>(p.num_seqs) * p.num_q_heads;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int64_t gr = row0 + 16 * warp + gq + 8 * hr;
    if (gr >= R) continue;
    const int64_t b = gr / p.group, j = gr % p.group;
    const int64_t hrow = split * stride + b * p.num_q_heads + g * p.group + j;
    float* dst = p.pf_o + hrow * D;
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      *reinterpret_cast<float2*>(dst + 8 * i + 2 * tq) = make_float2(o[i][2 * hr], o[i][2 * hr + 1]);
    if (tq == 0) p.pf_ml[hrow] = make_float2(m[hr], l[hr]);
  }
}

// Fold the S split partials of every (sequence, query head) row into the
// split-0 slot: M = max m_s, o = sum 2^(m_s - M) o_s, l = sum 2^(m_s - M)
// l_s.  One warp per row, lane l on columns 4l .. 4l+3 (and + 128 for
// D > 128); each lane reads its own columns of split 0 before writing them.
template <int D>
__global__ void __launch_bounds__(256) prefix_merge_kernel(const PrefixParams p) {
  pdl_wait();
  pdl_trigger();
  const int64_t rows = static_cast<int64_t>(p.num_seqs) * p.num_q_heads;
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float M = -INFINITY;
  for (int sp = 0; sp < p.splits; ++sp) M = fmaxf(M, p.pf_ml[sp * rows + row].x);
  float den = 0.f;
  float4 num[(D + 127) / 128];
#pragma unroll
  for (int j = 0; j < (D + 127) / 128; ++j) num[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int sp = 0; sp < p.splits; ++sp) {
    const float2 ml = p.pf_ml[sp * rows + row];
    const float w = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M);
    den = fmaf(w, ml.y, den);
#pragma unroll
    for (int j = 0; j < (D + 127) / 128; ++j) {
      const int d = 128 * j + 4 * lane;
      if (d < D) {
        const float4 x = *reinterpret_cast<const float4*>(p.pf_o + (sp * rows + row) * D + d);
        num[j].x = fmaf(w, x.x, num[j].x);
        num[j].y = fmaf(w, x.y, num[j].y);
        num[j].z = fmaf(w, x.z, num[j].z);
        num[j].w = fmaf(w, x.w, num[j].w);
      }
    }
  }
  __syncwarp();  // every lane has read split 0's (m, l)
#pragma unroll
  for (int j = 0; j < (D + 127) / 128; ++j) {
    const int d = 128 * j + 4 * lane;
    if (d < D) *reinterpret_cast<float4*>(p.pf_o + row * D + d) = num[j];
  }
  if (lane == 0) p.pf_ml[row] = make_float2(M, den);
}

}  // namespace pa
