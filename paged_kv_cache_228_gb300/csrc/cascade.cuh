// Shared-prefix pass of the cascade decode.
//
// "Paged Attention and KV Cache Fragmentation", section "How PagedAttention
// maps an OS concept onto GPU memory", and the "KV cache fragmentation"
// field guide, section "Why it matters": sequences forked from one prompt
// point at the same physical prefix blocks.  Attention over a sequence is
// the log-sum-exp merge of attention over any split of its tokens, so the
// prefix part can be computed once for every sequence's queries: for KV
// head g it is a dense product of all B*G query rows with the prefix keys
// and values, S = Q_g K_p^T, online softmax, O = P V_p.  The result is one
// partial (o unnormalised, m in log2 units, l) per (sequence, query head);
// the suffix decode and its merge fold it in.
//
// GB300 design: the two products run on the fifth-generation tensor cores
// (tcgen05.mma, kind::f16, M = 128 query rows, fp32 accumulators in tensor
// memory).  Q, K and V sit in shared memory in the 128-byte-swizzled layout
// the TMA writes.  A CTA makes each copied byte serve two 128-row query
// tiles: it owns 256 query rows of one KV head and one of S token ranges of
// the prefix, walked in 128-token chunks (N = 128 per score MMA: half the
// MMA instructions per token of 64-token chunks, and each instruction and
// each barrier round trip has a fixed cost).  Per query tile the tensor
// memory holds S of the chunk, overwritten in place by P (bf16, the A
// operand of the P.V product), and O.  Eleven warps:
//   warps 0/10 TMA producers of K and of V (one 2D box per block and
//              64-column slab) into K and V rings;
//   warp 1     owns the tensor memory; lane 0 issues the MMAs, per chunk j
//              and query tile t, once the softmax has written P_t,j:
//                O_t  += P_t,j . V_j                 (P in tensor memory,
//                                                     V MN-major; N = D)
//                S_t   = Q_t . K_j+1^T               (A, B K-major; N = 128)
//              in that order: the tensor pipe runs them in issue order, so
//              the scores of chunk j + 1 land in the columns of P_t,j only
//              after the product has read it, and their completion also
//              means the product is done;
//   warps 2-9  softmax, four warps per query tile, one row per thread (the
//              warp's quarter of the tensor-memory lanes): the chunk's
//              maximum in a first read of S, then 2^(s.scale - m) rounded to
//              bf16 pairs, written over S 32 columns at a time, and the sum
//              l of exactly those rounded weights.  The running max m moves,
//              and O_t is rescaled in tensor memory, only when a score
//              exceeds it by more than 8 in log2 units.  While one tile's
//              softmax runs, the tensor pipe works on the other tile.
// A negative scale is applied as its magnitude to the negated query (exact
// in bf16), so the maximum of a chunk is that of its raw scores.
// Each split writes its own partial per row (staged through shared memory
// so the global stores are coalesced); prefix_merge_kernel folds the S of
// them together.
#pragma once

#include "pa_device.cuh"
#include "umma.cuh"

namespace pa {

struct PrefixParams {
  const uint8_t* q;             // [num_seqs][num_q_heads][D] bf16
  const int32_t* prefix_table;  // the prefix's block ids (sequence 0's table)
  float* pf_o;                  // [splits][num_seqs * num_q_heads][D]
  float2* pf_ml;                // [splits][num_seqs * num_q_heads]
  int32_t num_seqs, num_q_heads, num_kv_heads, group, block_size, log2_bs, num_blocks;
  int32_t rows_total;     // num_blocks * num_kv_heads * block_size (rows of the K/V maps)
  int32_t prefix_tokens;
  int32_t prefix_chunks;  // ceil(prefix_tokens / kPfChunk)
  int32_t splits;         // S
  float scale_log2;
};

constexpr int kPfRows = 128;    // query rows per tile (the MMA's M)
constexpr int kPfTiles = 2;     // query tiles per CTA sharing each K/V chunk
constexpr int kPfChunk = 128;   // prefix tokens per chunk
constexpr int kPfKStages = 3;   // K ring depth
constexpr int kPfVStages = 2;   // V ring depth
constexpr int kPfSoftWarps = 4 * kPfTiles;
constexpr int kPfThreads = 96 + 32 * kPfSoftWarps;  // K and V producers, MMA, softmax
constexpr int kPfVWarp = 2 + kPfSoftWarps;
// Tensor memory per query tile (256 columns each): S of the chunk (128
// fp32, P in its first 64 columns once written), then O (D fp32).
constexpr int kPfTileCols = 256;
constexpr int kPfSCol = 0;
constexpr int kPfOCol = 128;
constexpr int kPfTmemCols = 512;
constexpr int kPfMaxSplits = 8;

template <int D>
struct PfSmem {
  static constexpr int kSlab = kPfChunk * 128;        // 64 columns of one chunk
  static constexpr int kKV = (D / 64) * kSlab;        // K (or V) of a chunk
  static constexpr int kQ = (D / 64) * kPfRows * 128; // one query tile
  static constexpr int kOffK = kPfTiles * kQ;
  static constexpr int kOffV = kOffK + kPfKStages * kKV;
  static constexpr int kOffBar = kOffV + kPfVStages * kKV;
  static constexpr int kBytes = kOffBar + 256;
  // the epilogue stages tile 0's partial in the (free) K ring, tile 1's in
  // the (free) V ring and the per-row (m, l) where Q was
  static_assert(kPfTiles == 2 && kPfRows * D * 4 <= kPfVStages * kKV &&
                    kPfRows * D * 4 <= kPfKStages * kKV,
                "epilogue staging");
  static_assert(kPfTiles * kPfRows * 8 <= kPfTiles * kQ, "epilogue (m, l)");
  static_assert(kPfSCol + kPfChunk <= kPfOCol && kPfOCol + D <= kPfTileCols,
                "tensor-memory columns");
  static_assert(kBytes <= 227 * 1024, "shared memory");
};

struct PfBars {
  uint64_t k_full[kPfKStages], k_empty[kPfKStages];
  uint64_t v_full[kPfVStages], v_empty[kPfVStages];
  uint64_t s_full[kPfTiles];  // S of the tile's chunk written (and its last product done)
  uint64_t p_full[kPfTiles];  // P of the tile's chunk written
  uint64_t o_last[kPfTiles];  // the tile's last product (and every MMA before it) done
  uint64_t mma_done;
  uint32_t tmem;
};
static_assert(sizeof(PfBars) <= 256, "barrier block");

// Byte offset of 16-byte chunk c (along the row's D * 2 bytes) of row r in
// a tile of `rows` rows stored as 128-byte slabs (128-byte swizzle).
__device__ __forceinline__ uint32_t pf_chunk(int rows, int r, int c) {
  return (c >> 3) * (rows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Producer lane i's block of chunk ch: the id of the block holding tokens
// [ch * kPfChunk + i * box_rows, + box_rows), or -1 past the prefix (and
// for lanes past the chunk's blocks).
__device__ __forceinline__ int32_t pf_block_id(const PrefixParams& p, int32_t ch) {
  const int lane = threadIdx.x & 31;
  const int box_rows = p.block_size < kPfChunk ? p.block_size : kPfChunk;
  const int32_t tok = ch * kPfChunk + lane * box_rows;
  if (lane >= kPfChunk / box_rows || tok >= p.prefix_tokens) return -1;
  return p.prefix_table[tok >> p.log2_bs];
}

// Producer lanes: the K (or V) rows of chunk ch into one ring stage, block i
// of the chunk (boxes of min(bs, 64) rows, one per 64-column slab) by lane
// i.  Blocks past the prefix, or with an invalid id, read rows past the
// tensor, which the TMA fills with zeros.
template <int D>
__device__ __forceinline__ void pf_copy_chunk(const PrefixParams& p, const CUtensorMap* map,
                                              int32_t g, int32_t ch, int32_t blk, uint32_t dst,
                                              uint32_t bar) {
  const int lane = threadIdx.x & 31;
  const int box_rows = p.block_size < kPfChunk ? p.block_size : kPfChunk;
  if (lane == 0) mbar_arrive_expect_tx(bar, PfSmem<D>::kKV);
  __syncwarp();
  if (lane < kPfChunk / box_rows) {
    const int32_t tok = ch * kPfChunk + lane * box_rows;
    int32_t row = p.rows_total;
    if (tok < p.prefix_tokens) {
      if (blk >= 0 && blk < p.num_blocks)
        row = (blk * p.num_kv_heads + g) * p.block_size + (tok & (p.block_size - 1));
      else
        flag_error(PA_DEVERR_BAD_BLOCK_ID);
    }
#pragma unroll
    for (int sl = 0; sl < D / 64; ++sl)
      tma_load_2d(dst + sl * PfSmem<D>::kSlab + lane * box_rows * 128, map, sl * 64, row, bar);
  }
}

// The largest raw score among 32 columns of a thread's row (chunk columns
// c0 .. c0 + 31), over those before `valid` when kMask, folded into `acc`.
// Two independent three-input maxima keep the chain short.
template <bool kMask>
__device__ __forceinline__ float pf_max32(const uint32_t (&u)[32], int32_t c0, int32_t valid,
                                          float acc) {
  auto v = [&](int i) {
    return !kMask || c0 + i < valid ? __uint_as_float(u[i]) : -INFINITY;
  };
  float a0 = acc, a1 = -INFINITY;
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    a0 = fmax3(a0, v(i), v(i + 1));
    a1 = fmax3(a1, v(i + 2), v(i + 3));
  }
  return fmaxf(a0, a1);
}

// The weights 2^(s * sl - m) (neg = -m) of 32 columns, rounded to bf16
// pairs: w[c] holds columns 2c (low half) and 2c + 1, the layout of the
// P.V product's A operand in tensor memory; columns from `valid` on weigh
// 0 when kMask.  l (one sum per half of the pairs) gains the sum of the
// rounded weights.
template <bool kMask>
__device__ __forceinline__ void pf_weights32(const uint32_t (&u)[32], int32_t c0, int32_t valid,
                                             float sl, float neg, uint32_t (&w)[16], float2& l) {
  const float2 s2 = make_float2(sl, sl), n2 = make_float2(neg, neg);
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const float2 x =
        fma2(make_float2(__uint_as_float(u[2 * c]), __uint_as_float(u[2 * c + 1])), s2, n2);
    float e0 = fast_exp2(x.x), e1 = fast_exp2(x.y);
    if (kMask) {
      e0 = c0 + 2 * c < valid ? e0 : 0.f;
      e1 = c0 + 2 * c + 1 < valid ? e1 : 0.f;
    }
    w[c] = pack_bf16x2(e0, e1);
    l = add2(l, unpack_bf16x2(w[c]));
  }
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefix_attention_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const PrefixParams p) {
  using L = PfSmem<D>;
  extern __shared__ __align__(1024) uint8_t pf_smem[];
  const uint32_t base = smem_addr(pf_smem);
  if (base & 1023u) {  // the same for every CTA of the launch
    if (threadIdx.x == 0) flag_error(PA_DEVERR_LAUNCH);
    return;
  }
  PfBars* bars = reinterpret_cast<PfBars*>(pf_smem + L::kOffBar);
  const uint32_t sq = base, sk = base + L::kOffK, sv = base + L::kOffV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t g = blockIdx.y, split = blockIdx.z;
  const uint32_t G = static_cast<uint32_t>(p.group);
  const uint32_t R = static_cast<uint32_t>(p.num_seqs) * G;  // query rows of head g
  const uint32_t row0 = blockIdx.x * (kPfTiles * kPfRows);
  const int32_t c0 = static_cast<int32_t>(static_cast<int64_t>(p.prefix_chunks) * split / p.splits);
  const int32_t c1 = static_cast<int32_t>(static_cast<int64_t>(p.prefix_chunks) * (split + 1) / p.splits);
  const int32_t n = c1 - c0;
  // The CTAs of one token range (one per 256 query rows) walk its chunks
  // from different starting points, so that they do not all ask for the
  // same lines at the same moment; the log-sum-exp fold is order-free.
  const int32_t rot = n > 0 ? static_cast<int32_t>(static_cast<int64_t>(blockIdx.x) * n / gridDim.x) : 0;
  auto chunk = [&](int32_t j) -> int32_t { return c0 + (j + rot < n ? j + rot : j + rot - n); };
  // q / partial row of CTA row r (r < R - row0): sequence b, head g*G + j
  auto head_row = [&](uint32_t r) -> int64_t {
    const uint32_t gr = row0 + r, b = gr / G, j = gr - b * G;
    return static_cast<int64_t>(b) * p.num_q_heads + g * p.group + j;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPfKStages; ++i) {
      mbar_init(smem_addr(&bars->k_full[i]), 1);
      mbar_init(smem_addr(&bars->k_empty[i]), 1);
    }
    for (int i = 0; i < kPfVStages; ++i) {
      mbar_init(smem_addr(&bars->v_full[i]), 1);
      mbar_init(smem_addr(&bars->v_empty[i]), 1);
    }
    for (int t = 0; t < kPfTiles; ++t) {
      mbar_init(smem_addr(&bars->s_full[t]), 1);
      mbar_init(smem_addr(&bars->p_full[t]), 4);
      mbar_init(smem_addr(&bars->o_last[t]), 1);
    }
    mbar_init(smem_addr(&bars->mma_done), 1);
    mbar_fence_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncthreads();  // barriers initialised
  pdl_wait();       // launched as a programmatic dependent: inputs ready below
  pdl_trigger();
  bool ok = true;
  uint32_t tmem = 0;
  if (warp >= 1 && warp < kPfVWarp) {
    // The tensor memory (warp 1) and the 256 query rows (softmax warps;
    // zeros past R, negated for a negative scale), then a barrier of warps
    // 1-9.  The producers have started meanwhile.
    if (warp == 1) {
      tmem_alloc(smem_addr(&bars->tmem), kPfTmemCols);
      tmem_relinquish();
    } else {
      constexpr int kCpr = D * 2 / 16;
      constexpr int kSoft = 32 * kPfSoftWarps;
      constexpr int kPer = kPfTiles * kPfRows * kCpr / kSoft;  // 16-byte chunks per thread
      const uint32_t flip = p.scale_log2 < 0.f ? 0x80008000u : 0u;
      const int t = threadIdx.x - 64;
      uint4 v[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {  // all loads in flight first
        const int idx = t + kSoft * i, r = idx / kCpr, c = idx % kCpr;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (row0 + r < R)
          v[i] = *reinterpret_cast<const uint4*>(p.q + head_row(r) * (D * 2) + c * 16);
      }
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int idx = t + kSoft * i, r = idx / kCpr, c = idx % kCpr;
        const uint32_t a = sq + (r / kPfRows) * L::kQ + pf_chunk(kPfRows, r % kPfRows, c);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v[i].x ^ flip),
                     "r"(v[i].y ^ flip), "r"(v[i].z ^ flip), "r"(v[i].w ^ flip)
                     : "memory");
      }
      fence_proxy_async_smem();  // the MMA (async proxy) reads Q
    }
    tc_fence_before_sync();
    asm volatile("bar.sync 1, %0;" ::"r"(32 * (kPfVWarp - 1)) : "memory");
    tc_fence_after_sync();
    tmem = bars->tmem;
  }

  if (warp == 0 || warp == kPfVWarp) {
    // ----------------------------------------- producers: K (0), V (10) ---
    const bool is_k = warp == 0;
    const int S = is_k ? kPfKStages : kPfVStages;
    const CUtensorMap* map = is_k ? &tm_k : &tm_v;
    const uint32_t ring = is_k ? sk : sv;
    uint64_t* full = is_k ? bars->k_full : bars->v_full;
    uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
    int32_t issued = 0;
    int32_t e = n > 0 ? pf_block_id(p, chunk(0)) : -1, en = n > 1 ? pf_block_id(p, chunk(1)) : -1;
    for (int32_t j = 0; j < n && ok; ++j) {
      const int st = j % S;
      if (lane == 0 && j >= S) ok = mbar_wait(smem_addr(&empty[st]), ((j / S) - 1) & 1);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      pf_copy_chunk<D>(p, map, g, chunk(j), e, ring + st * L::kKV, smem_addr(&full[st]));
      issued = j + 1;
      e = en;  // the next chunk's ids, loaded a chunk ahead
      en = j + 2 < n ? pf_block_id(p, chunk(j + 2)) : -1;
    }
    // No copy may still target shared memory when the CTA exits: on the
    // normal path the MMAs have consumed every one already.
    if (lane == 0)
      for (int32_t j = issued > S ? issued - S : 0; j < issued; ++j)
        mbar_wait(smem_addr(&full[j % S]), (j / S) & 1, 1u << 16);
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16(kPfRows, kPfChunk, false, false);
      constexpr uint32_t kIdPV = idesc_bf16(kPfRows, D, false, true);
      // S_t = Q_t . K^T of the chunk whose K sits at kb
      auto qk = [&](int t, uint32_t kb) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * (kPfRows * 128) + (k & 3) * 32;
          const uint32_t koff = (k >> 2) * L::kSlab + (k & 3) * 32;
          umma_bf16(tmem + t * kPfTileCols + kPfSCol,
                    smem_desc_sw128(sq + t * L::kQ + off, 16, 1024),
                    smem_desc_sw128(kb + koff, 16, 1024), kIdQK, k > 0);
        }
        umma_commit(smem_addr(&bars->s_full[t]));
      };
      if (n > 0) {
        ok = mbar_wait(smem_addr(&bars->k_full[0]), 0);
        if (ok) {
          tc_fence_after_sync();
          for (int t = 0; t < kPfTiles; ++t) qk(t, sk);
          umma_commit(smem_addr(&bars->k_empty[0]));
        }
      }
      uint32_t last = 0;  // tiles whose o_last has been committed
      for (int32_t j = 0; j < n && ok; ++j) {
        const int vs = j % kPfVStages, ks = (j + 1) % kPfKStages;
        const bool more = j + 1 < n;
        const uint32_t vb = sv + vs * L::kKV, kb = sk + ks * L::kKV;
        ok = mbar_wait(smem_addr(&bars->v_full[vs]), (j / kPfVStages) & 1);
        for (int t = 0; t < kPfTiles && ok; ++t) {
          // P_t of chunk j written (over S_t); then its product and the
          // scores of chunk j + 1, in that order
          ok = mbar_wait(smem_addr(&bars->p_full[t]), j & 1);
          if (ok && more && t == 0)
            ok = mbar_wait(smem_addr(&bars->k_full[ks]), ((j + 1) / kPfKStages) & 1);
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t tt = tmem + t * kPfTileCols;
#pragma unroll
          for (int k = 0; k < kPfChunk / 16; ++k)
            umma_bf16_ta(tt + kPfOCol, tt + kPfSCol + k * 8,
                         smem_desc_sw128(vb + k * 16 * 128, L::kSlab, 1024), kIdPV,
                         j > 0 || k > 0);
          if (more) {
            qk(t, kb);
          } else {
            umma_commit(smem_addr(&bars->o_last[t]));
            last |= 1u << t;
          }
        }
        if (!ok) break;
        umma_commit(smem_addr(&bars->v_empty[vs]));
        if (more) umma_commit(smem_addr(&bars->k_empty[ks]));
      }
      // a wait that failed still releases the softmax warps
      for (int t = 0; t < kPfTiles; ++t)
        if (!(last >> t & 1u)) umma_commit(smem_addr(&bars->o_last[t]));
      // every MMA this thread issued has completed before the tensor
      // memory is released
      umma_commit(smem_addr(&bars->mma_done));
      mbar_wait(smem_addr(&bars->mma_done), 0, 1u << 16);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- softmax ---
    const int tile = (warp - 2) >> 2;
    const int quarter = warp & 3;  // tensor-memory lanes 32 * quarter ...
    const int r = 32 * quarter + lane;  // row within the tile
    const uint32_t tb =
        tmem + (static_cast<uint32_t>(32 * quarter) << 16) + tile * kPfTileCols;
    const float sl = fabsf(p.scale_log2);
    float m = -INFINITY;
    float2 l = make_float2(0.f, 0.f);
    for (int32_t j = 0; j < n; ++j) {
      ok = mbar_wait(smem_addr(&bars->s_full[tile]), j & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int32_t valid = p.prefix_tokens - chunk(j) * kPfChunk;  // tokens of the chunk
      const bool part = valid < kPfChunk;  // the prefix's last, partial chunk
      // pass 1: the chunk's largest score
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < kPfChunk / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tb + kPfSCol + 32 * c, u);
        tmem_wait_ld();
        mx = part ? pf_max32<true>(u, 32 * c, valid, mx) : pf_max32<false>(u, 32 * c, valid, mx);
      }
      mx *= sl;
      if (j == 0) {
        m = mx;
      } else if (__any_sync(0xffffffffu, mx > m + 8.f)) {
        // the running max moves: O and l scale by alpha.  O holds the
        // products through chunk j - 1, all complete (the scores of chunk
        // j were issued after them), and the product of chunk j waits for
        // this warp's P.
        const float mn = fmaxf(m, mx);
        const float alpha = fast_exp2(m - mn);
        m = mn;
        l.x *= alpha;
        l.y *= alpha;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t u[32];
          tmem_ld32(tb + kPfOCol + 32 * c, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
          tmem_st32(tb + kPfOCol + 32 * c, u);
        }
      }
      // pass 2: P over the first half of S, 32 scores (16 columns of P) at
      // a time; P's columns 16c .. 16c + 15 lie among scores already read
      const float neg = -m;
#pragma unroll 1
      for (int c = 0; c < kPfChunk / 32; ++c) {
        uint32_t u[32], w[16];
        tmem_ld32(tb + kPfSCol + 32 * c, u);
        tmem_wait_ld();
        if (part)
          pf_weights32<true>(u, 32 * c, valid, sl, neg, w, l);
        else
          pf_weights32<false>(u, 32 * c, valid, sl, neg, w, l);
        tmem_st16(tb + kPfSCol + 16 * c, w);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bars->p_full[tile]));
    }
    // this tile's last product is complete, and with it every score MMA
    // (issued before it) and the other tile's products but its last one: the
    // K ring and Q's room are free, the V ring once the other tile is done
    ok = mbar_wait(smem_addr(&bars->o_last[tile]), 0) && ok;
    ok = __all_sync(0xffffffffu, ok);
    // (m, l) of each row where Q was
    reinterpret_cast<float2*>(pf_smem)[tile * kPfRows + r] = make_float2(m, l.x + l.y);
  }
  // ---- epilogue, each tile as soon as its last product is done: its
  // rows' partials (o unnormalised) are staged in shared memory (tile 0 in
  // the K ring, tile 1 in the V ring; float rows of D, 16-byte chunk c of
  // row r at chunk c ^ (r % (D/4))), then written to this split's slot with
  // coalesced stores by the tile's four warps (warp w of the tile rows w,
  // w + 4, ...; lane l its 16-byte chunk).
  constexpr int kCh = D / 4;
  const int64_t slot = static_cast<int64_t>(split) * p.num_seqs * p.num_q_heads;
  if (warp >= 2 && warp < kPfVWarp) {
    const int t = (warp - 2) >> 2, quarter = warp & 3, r = 32 * quarter + lane;
    const uint32_t stage_addr = t == 0 ? sk : sv;
    const bool go = ok && n > 0;
    if (go) {
      const uint32_t tb = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + t * kPfTileCols;
      tc_fence_after_sync();
#pragma unroll
      for (int part = 0; part < D / 32; ++part) {
        uint32_t u[32];
        tmem_ld32(tb + kPfOCol + part * 32, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = part * 8 + i;
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(
                           stage_addr + (r * D + 4 * (c ^ (r & (kCh - 1)))) * 4),
                       "r"(u[4 * i]), "r"(u[4 * i + 1]), "r"(u[4 * i + 2]), "r"(u[4 * i + 3])
                       : "memory");
        }
      }
      if (row0 + t * kPfRows + r < R)
        p.pf_ml[slot + head_row(t * kPfRows + r)] =
            reinterpret_cast<const float2*>(pf_smem)[t * kPfRows + r];
    }
    if (t == 0)
      asm volatile("bar.sync 2, 128;" ::: "memory");
    else
      asm volatile("bar.sync 3, 128;" ::: "memory");
    if (go && lane < kCh) {
      for (int r2 = quarter; r2 < kPfRows && row0 + t * kPfRows + r2 < R; r2 += 4) {
        float4 x;
        asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                     : "r"(stage_addr + (r2 * D + 4 * (lane ^ (r2 & (kCh - 1)))) * 4)
                     : "memory");
        reinterpret_cast<float4*>(p.pf_o + (slot + head_row(t * kPfRows + r2)) * D)[lane] = x;
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kPfTmemCols);
  }
}

// Fold the S split partials of every (sequence, query head) row into the
// split-0 slot: M = max m_s, o = sum 2^(m_s - M) o_s, l = sum 2^(m_s - M)
// l_s.  One thread per (row, 16-byte chunk of the row); its loads of all
// splits are issued together (S <= kPfMaxSplits), and it reads split 0's
// chunk before writing it.
template <int D>
__global__ void __launch_bounds__(256) prefix_merge_kernel(const PrefixParams p) {
  pdl_wait();
  pdl_trigger();
  constexpr int kCh = D / 4;
  const int64_t rows = static_cast<int64_t>(p.num_seqs) * p.num_q_heads;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = idx / kCh;
  const int c = static_cast<int>(idx % kCh);
  if (row >= rows) return;
  float2 ml[kPfMaxSplits];
  float4 x[kPfMaxSplits];
#pragma unroll
  for (int sp = 0; sp < kPfMaxSplits; ++sp)
    if (sp < p.splits) {
      ml[sp] = p.pf_ml[sp * rows + row];
      x[sp] = reinterpret_cast<const float4*>(p.pf_o + (sp * rows + row) * D)[c];
    }
  float M = -INFINITY;
#pragma unroll
  for (int sp = 0; sp < kPfMaxSplits; ++sp)
    if (sp < p.splits) M = fmaxf(M, ml[sp].x);
  float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
#pragma unroll
  for (int sp = 0; sp < kPfMaxSplits; ++sp)
    if (sp < p.splits) {
      const float w = fast_exp2(ml[sp].x - M);
      den = fmaf(w, ml[sp].y, den);
      num.x = fmaf(w, x[sp].x, num.x);
      num.y = fmaf(w, x[sp].y, num.y);
      num.z = fmaf(w, x[sp].z, num.z);
      num.w = fmaf(w, x[sp].w, num.w);
    }
  reinterpret_cast<float4*>(p.pf_o + row * D)[c] = num;
  // every thread of the row has read split 0's (m, l) before it changes:
  // the row's kCh threads are consecutive, aligned lanes of one warp
  __syncwarp(kCh == 32 ? 0xffffffffu : (((1u << kCh) - 1u) << (threadIdx.x & (32 - kCh))));
  if (c == 0) p.pf_ml[row] = make_float2(M, den);
}

}  // namespace pa
