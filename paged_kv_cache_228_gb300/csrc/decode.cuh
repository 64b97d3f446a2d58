// Paged single-token decode attention for sm_103a.
//
// Method: "KV cache fragmentation" (field guide), section "Definition" -- the
// attention kernel walks a per-request table from logical position to
// physical page; "Paged Attention and KV Cache Fragmentation", section "How
// PagedAttention maps an OS concept onto GPU memory" -- fixed-size blocks, a
// request sees one continuous sequence.  The result is dense attention over
// the logical sequence, softmax(scale * q K^T) V, accumulated in fp32
// (section "Quantization as a way to stretch paged memory further" for the
// FP8 cache and the fp32 accumulation it needs).
//
// GB300 design
// ------------
// * Work unit: a 16-token tile of one (sequence b, KV head g) "segment".
//   All tiles of all segments form one flat list of W tiles, ordered
//   (b, g, tile); persistent CTA c of P owns tiles [W*c/P, W*(c+1)/P).  This
//   balances ragged lengths to within one tile per CTA and splits long
//   contexts into at most P pieces in total (split-K).  A piece that covers
//   a whole segment writes the output directly; otherwise it writes an
//   unnormalised partial (o, m, l) that the merge kernel combines by
//   log-sum-exp.  Split points depend only on seq_lens, so the output does
//   not depend on which physical blocks the tables name.
// * CTA = 2 warps.  Warp 0 (producer) reads block-table entries 32 at a
//   time with one coalesced warp load and issues 2D TMA copies of each
//   tile's K and V rows (128-byte wide boxes, 128B swizzle) into a ring of
//   shared-memory stages guarded by mbarriers; it also stages the G query
//   rows of each new segment.  Warp 1 (consumer) runs the math.  Several
//   CTAs per SM keep >100 KB of loads in flight per SM.
// * Math on tensor cores (mma.sync m16n8k16, fp32 accumulate), tokens on M
//   and the GQA group on N, so one K/V tile feeds every query head of its
//   group from a single read:
//     S^T[16 tok x 8 heads] = K_tile[16 x d] . Q^T[d x 8]     (ldmatrix)
//     online softmax per head column in fp32 (running max m, sum l)
//     O^T[d x 8 heads]     += V_tile^T[d x 16] . P^T[16 x 8] (ldmatrix.trans)
//   P^T's fragment comes from S^T's accumulator by one movmatrix.trans per
//   8x8 quarter.  FP8 tiles: QK runs on the E4M3 MMA straight from the
//   cache bytes (the query as a two-term E4M3 split), PV on the f16 MMA
//   with V converted exactly in registers; the per-(block, head) K scale
//   multiplies the scores and the V scale the per-tile P.V product, so
//   accumulation stays fp32.
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kTile = 16;  // tokens per work tile
constexpr int kMaxG = 8;   // query heads per KV head handled by one N=8 MMA

struct DecodeParams {
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const float* k_scale;
  const float* v_scale;
  __nv_bfloat16* out;
  float* ws_o;    // [pieces][kMaxG][D] unnormalised partial outputs
  float2* ws_ml;  // [pieces][kMaxG] (running max in log2 units, sum)
  int32_t num_seqs, num_q_heads, num_kv_heads, group, block_size, log2_bs;
  int32_t max_blocks, num_blocks;
  int32_t rows_total;  // num_blocks * num_kv_heads * block_size
  float scale_log2;    // softmax scale * log2(e)
  int32_t num_ctas;    // P
  int32_t stages;      // ring depth
};

// ------------------------------------------------ shared memory layout ---
template <int D, bool FP8>
struct Smem {
  static constexpr int kSlabBytes = FP8 ? kTile * D : kTile * 128;  // one box
  static constexpr int kSlabs = FP8 ? 1 : D / 64;
  static constexpr int kKVBytes = kSlabs * kSlabBytes;  // K (or V) of a tile
  static constexpr int kStageBytes = 2 * kKVBytes;
  static constexpr int kQSlabBytes = 8 * 128;           // 8 rows x 64 bf16
  static constexpr int kQBytes = (D / 64) * kQSlabBytes;
  static constexpr int kHeaderBytes = 1024;  // barriers + per-stage scales
  static constexpr int kMaxStages = 24;
};

struct Header {
  uint64_t full[24];
  uint64_t empty[24];
  uint64_t qfull[2];
  uint64_t qempty[2];
  float4 scales[24];  // FP8: (k_scale row g, k_scale row g+8, v_scale ...)
};
static_assert(sizeof(Header) <= 1024, "header overflow");

__device__ __forceinline__ int32_t cdiv16(int32_t n) { return (n + 15) >> 4; }

__device__ __forceinline__ int32_t clamp_len(const DecodeParams& p, int32_t n) {
  const int32_t cap = p.max_blocks * p.block_size;
  if (n < 0 || n > cap) {
    flag_error(PA_DEVERR_BAD_SEQ_LEN);
    n = n < 0 ? 0 : cap;
  }
  return n;
}

// Position in the flat tile list: segment (b, g), tile within it.
struct Cursor {
  int32_t b, g, tile, T, n;
};

// Warp-collective: find the segment holding flat tile u (< W).
__device__ __forceinline__ void locate(const DecodeParams& p, int64_t u,
                                       Cursor& c) {
  const int lane = threadIdx.x & 31;
  int64_t base = 0;
  for (int32_t b0 = 0; b0 < p.num_seqs; b0 += 32) {
    const int32_t b = b0 + lane;
    const int32_t n = b < p.num_seqs ? clamp_len(p, p.seq_lens[b]) : 0;
    const int64_t w = static_cast<int64_t>(p.num_kv_heads) * cdiv16(n);
    int64_t incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int64_t total = __shfl_sync(0xffffffffu, incl, 31);
    if (base + total > u) {
      const unsigned m = __ballot_sync(0xffffffffu, base + incl > u);
      const int L = __ffs(m) - 1;
      const int64_t excl = __shfl_sync(0xffffffffu, incl - w, L);
      const int32_t nn = __shfl_sync(0xffffffffu, n, L);
      const int64_t rem = u - (base + excl);
      c.b = b0 + L;
      c.n = nn;
      c.T = cdiv16(nn);
      c.g = static_cast<int32_t>(rem / c.T);
      c.tile = static_cast<int32_t>(rem % c.T);
      return;
    }
    base += total;
  }
  c.b = p.num_seqs;  // unreachable for u < W
  c.g = c.tile = c.T = c.n = 0;
}

// Move to the first tile of the next non-empty segment.
__device__ __forceinline__ void next_segment(const DecodeParams& p, Cursor& c) {
  c.tile = 0;
  if (++c.g < p.num_kv_heads) return;
  c.g = 0;
  do {
    ++c.b;
    c.n = c.b < p.num_seqs ? clamp_len(p, p.seq_lens[c.b]) : 1;
    c.T = cdiv16(c.n);
  } while (c.T == 0);
}

// Flat-list range of CTA c of P (P <= W, so every range is non-empty).
__device__ __forceinline__ void cta_range(int64_t W, int32_t P, int32_t c,
                                          int64_t& lo, int64_t& hi) {
  lo = W * c / P;
  hi = W * (c + 1) / P;
}

// Index of the CTA whose range holds flat tile u.
__device__ __forceinline__ int32_t cta_of(int64_t W, int32_t P, int64_t u) {
  return static_cast<int32_t>(((u + 1) * P - 1) / W);
}

// Warp-collective total tile count W.
__device__ __forceinline__ int64_t total_tiles(const DecodeParams& p) {
  const int lane = threadIdx.x & 31;
  int64_t w = 0;
  for (int32_t b = lane; b < p.num_seqs; b += 32)
    w += cdiv16(clamp_len(p, p.seq_lens[b]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
  return w * p.num_kv_heads;
}

// ------------------------------------------------------------ producer ---
template <int D, bool FP8>
__device__ __forceinline__ void producer(const DecodeParams& p,
                                         const CUtensorMap* tm_q,
                                         const CUtensorMap* tm_k,
                                         const CUtensorMap* tm_v, Header* hdr,
                                         uint32_t qbuf, uint32_t ring,
                                         int64_t lo, int64_t hi) {
  using L = Smem<D, FP8>;
  const int lane = threadIdx.x & 31;
  Cursor c;
  locate(p, lo, c);
  int64_t u = lo;
  uint32_t it = 0;      // tiles issued
  uint32_t qcount = 0;  // segments issued
  const int box_rows = p.block_size < kTile ? p.block_size : kTile;
  const uint32_t box_bytes = static_cast<uint32_t>(box_rows) * (FP8 ? D : 128);
  bool ok = true;
  while (u < hi && ok) {
    const int32_t seg_end = static_cast<int32_t>(
        min(static_cast<int64_t>(c.T), c.tile + (hi - u)));
    // Query rows of this segment: 8 rows from b*Hq + g*G (rows past the
    // group are ignored by the consumer; past the tensor they read zeros).
    if (lane == 0) {
      const uint32_t slot = qcount & 1;
      if (qcount >= 2) ok = mbar_wait(smem_addr(&hdr->qempty[slot]), ((qcount >> 1) - 1) & 1);
      if (ok) {
        const uint32_t bar = smem_addr(&hdr->qfull[slot]);
        mbar_arrive_expect_tx(bar, L::kQBytes);
        const int32_t row = c.b * p.num_q_heads + c.g * p.group;
#pragma unroll
        for (int s = 0; s < D / 64; ++s)
          tma_load_2d(qbuf + slot * L::kQBytes + s * L::kQSlabBytes, tm_q,
                      s * 64, row, bar);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    ++qcount;
    const int32_t* trow = p.block_tables + static_cast<int64_t>(c.b) * p.max_blocks;
    const int32_t kvrow_base = c.g;  // row = (blk * Hkv + g) * bs + offset
    for (int32_t t0 = c.tile; t0 < seg_end && ok; t0 += 32) {
      const int32_t nt = min(32, seg_end - t0);
      // One coalesced load of the table entries of up to 32 tiles.
      int32_t e0 = -1, e1 = -1;
      float ks0 = 1.f, ks1 = 1.f, vs0 = 1.f, vs1 = 1.f;
      if (lane < nt) {
        const int32_t tok = (t0 + lane) * kTile;
        if (p.block_size >= kTile) {
          e0 = trow[tok >> p.log2_bs];
        } else {
          e0 = trow[tok >> p.log2_bs];
          if (tok + p.block_size < c.n) e1 = trow[(tok >> p.log2_bs) + 1];
        }
        bool bad = e0 < 0 || e0 >= p.num_blocks;
        if (p.block_size < kTile && tok + p.block_size < c.n)
          bad |= e1 < 0 || e1 >= p.num_blocks;
        if (bad) flag_error(PA_DEVERR_BAD_BLOCK_ID);
        if (FP8) {
          if (e0 >= 0 && e0 < p.num_blocks) {
            ks0 = p.k_scale[static_cast<int64_t>(e0) * p.num_kv_heads + c.g];
            vs0 = p.v_scale[static_cast<int64_t>(e0) * p.num_kv_heads + c.g];
          }
          ks1 = ks0;
          vs1 = vs0;
          if (p.block_size < kTile && e1 >= 0 && e1 < p.num_blocks) {
            ks1 = p.k_scale[static_cast<int64_t>(e1) * p.num_kv_heads + c.g];
            vs1 = p.v_scale[static_cast<int64_t>(e1) * p.num_kv_heads + c.g];
          }
        }
      }
      for (int32_t j = 0; j < nt; ++j) {
        const int32_t b0 = __shfl_sync(0xffffffffu, e0, j);
        const int32_t b1 = __shfl_sync(0xffffffffu, e1, j);
        float4 sc;
        sc.x = __shfl_sync(0xffffffffu, ks0, j);
        sc.y = __shfl_sync(0xffffffffu, ks1, j);
        sc.z = __shfl_sync(0xffffffffu, vs0, j);
        sc.w = __shfl_sync(0xffffffffu, vs1, j);
        if (lane == 0) {
          const uint32_t stage = it % p.stages;
          const uint32_t use = it / p.stages;
          if (use > 0) ok = mbar_wait(smem_addr(&hdr->empty[stage]), (use - 1) & 1);
          if (ok) {
            if (FP8) hdr->scales[stage] = sc;
            const int32_t tile = t0 + j;
            const int32_t tok = tile * kTile;
            const int nbox = (p.block_size < kTile && tok + p.block_size < c.n) ? 2 : 1;
            const uint32_t bar = smem_addr(&hdr->full[stage]);
            mbar_arrive_expect_tx(bar, 2u * nbox * L::kSlabs * box_bytes);
            const uint32_t kdst = ring + stage * L::kStageBytes;
            const uint32_t vdst = kdst + L::kKVBytes;
            for (int bx = 0; bx < nbox; ++bx) {
              const int32_t blk = bx == 0 ? b0 : b1;
              int32_t row;
              if (blk < 0 || blk >= p.num_blocks) {
                row = p.rows_total;  // out of the tensor: TMA fills zeros
              } else {
                const int32_t off = p.block_size >= kTile ? (tok & (p.block_size - 1)) : 0;
                row = (blk * p.num_kv_heads + kvrow_base) * p.block_size + off;
              }
              const uint32_t sub = static_cast<uint32_t>(bx) * box_bytes;
#pragma unroll
              for (int s = 0; s < L::kSlabs; ++s) {
                tma_load_2d(kdst + s * L::kSlabBytes + sub, tm_k, s * 64, row, bar);
                tma_load_2d(vdst + s * L::kSlabBytes + sub, tm_v, s * 64, row, bar);
              }
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        ++it;
        if (!ok) break;
      }
    }
    u += seg_end - c.tile;
    if (u < hi) next_segment(p, c);
  }
  // Drain: wait until every copy this CTA issued has landed (no TMA may
  // target shared memory after the CTA exits).  On the normal path the
  // consumer already waited for all of them.
  if (lane == 0) {
    const uint32_t S = p.stages;
    const uint32_t first = it > S ? it - S : 0;
    for (uint32_t k = first; k < it; ++k)
      mbar_wait(smem_addr(&hdr->full[k % S]), (k / S) & 1, 1u << 16);
    for (uint32_t k = (qcount > 2 ? qcount - 2 : 0); k < qcount; ++k)
      mbar_wait(smem_addr(&hdr->qfull[k & 1]), (k >> 1) & 1, 1u << 16);
  }
}

// ------------------------------------------------------------ consumer ---
// Lane (gq = lane / 4, tq = lane % 4) owns, in every m16n8 fragment, rows
// gq and gq + 8 and columns 2tq, 2tq + 1 (heads).
template <int D>
struct SegState {
  float acc[D / 16][4];  // O^T fragments: (d = 16i + gq [+8], heads 2tq, 2tq+1)
  float m[2];            // running max (log2 units) of heads 2tq, 2tq+1
  float l[2];            // this lane's share of the running sum
};

template <int D>
__device__ __forceinline__ void seg_reset(SegState<D>& s) {
#pragma unroll
  for (int i = 0; i < D / 16; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) s.acc[i][j] = 0.f;
  s.m[0] = s.m[1] = -INFINITY;
  s.l[0] = s.l[1] = 0.f;
}

// Online-softmax update from one tile's scores (already in log2 units and
// masked); returns P packed for the PV MMA B operand (b0: tokens 0-7,
// b1: tokens 8-15) and the rescale factors.
template <bool F16P>
__device__ __forceinline__ void softmax_tile(float x0, float x1, float x2,
                                             float x3, float (&m)[2],
                                             float (&l)[2], float ratio0,
                                             float ratio1, float& alpha0,
                                             float& alpha1, uint32_t& pb0,
                                             uint32_t& pb1) {
  // Conditional rescaling: the running max only moves when some score of
  // the tile exceeds it by more than kSlack (log2 units); otherwise the
  // weights 2^(x - m) stay <= 2^kSlack, exact enough in bf16/f16 and summed
  // in fp32, and the cross-lane max reduction is skipped.  The first tile of
  // a segment (m = -inf) always takes the full path.
  constexpr float kSlack = 8.f;
  const bool grow = fmaxf(x0, x2) > m[0] + kSlack || fmaxf(x1, x3) > m[1] + kSlack;
  alpha0 = alpha1 = 1.f;
  if (__any_sync(0xffffffffu, grow)) {
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
    alpha0 = fast_exp2(m[0] - mn0);
    alpha1 = fast_exp2(m[1] - mn1);
    m[0] = mn0;
    m[1] = mn1;
  }
  const float p0 = fast_exp2(x0 - m[0]), p1 = fast_exp2(x1 - m[1]);
  const float p2 = fast_exp2(x2 - m[0]), p3 = fast_exp2(x3 - m[1]);
  uint32_t P01, P23;
  float2 r01, r23;
  if (F16P) {
    P01 = pack_f16x2(p0 * ratio0, p1 * ratio0);
    P23 = pack_f16x2(p2 * ratio1, p3 * ratio1);
    r01 = make_float2(p0, p1);
    r23 = make_float2(p2, p3);
  } else {
    P01 = pack_bf16x2(p0, p1);
    P23 = pack_bf16x2(p2, p3);
    r01 = unpack_bf16x2(P01);  // sum exactly the weights the MMA applies
    r23 = unpack_bf16x2(P23);
  }
  l[0] = l[0] * alpha0 + (r01.x + r23.x);
  l[1] = l[1] * alpha1 + (r01.y + r23.y);
  pb0 = movmatrix_t(P01);
  pb1 = movmatrix_t(P23);
}

template <int D>
__device__ __forceinline__ void rescale(SegState<D>& s, float alpha0,
                                        float alpha1) {
  const bool need = __any_sync(0xffffffffu, alpha0 != 1.f || alpha1 != 1.f);
  if (!need) return;
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    s.acc[i][0] *= alpha0;
    s.acc[i][1] *= alpha1;
    s.acc[i][2] *= alpha0;
    s.acc[i][3] *= alpha1;
  }
}

// bf16 tile: K/V slabs of 16 rows x 128 B, 128B swizzle.
template <int D>
__device__ __forceinline__ void tile_bf16(const DecodeParams& p, uint32_t kb,
                                          uint32_t vb, int valid,
                                          const uint32_t (&qb)[D / 16][2],
                                          SegState<D>& s) {
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2;
  // S^T = K . Q^T, two interleaved accumulators to halve the MMA chain.
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t rowaddr = kb + r * 128;
    const int rx = r & 7;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int ch = (kk & 3) * 2 + (lane >> 4);
      uint32_t a0, a1, a2, a3;
      ldsm_x4(rowaddr + (kk >> 2) * 2048 + ((ch ^ rx) << 4), a0, a1, a2, a3);
      if (kk & 1)
        mma_bf16(sb, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      else
        mma_bf16(sa, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
    }
  }
  float x0 = (sa[0] + sb[0]) * p.scale_log2, x1 = (sa[1] + sb[1]) * p.scale_log2;
  float x2 = (sa[2] + sb[2]) * p.scale_log2, x3 = (sa[3] + sb[3]) * p.scale_log2;
  if (gq >= valid) x0 = x1 = -INFINITY;
  if (gq + 8 >= valid) x2 = x3 = -INFINITY;
  float alpha0, alpha1;
  uint32_t pb0, pb1;
  softmax_tile<false>(x0, x1, x2, x3, s.m, s.l, 1.f, 1.f, alpha0, alpha1, pb0, pb1);
  rescale(s, alpha0, alpha1);
  // O^T += V^T . P^T
  {
    const int j = lane >> 3;
    const int r = (lane & 7) + (j >> 1) * 8;
    const uint32_t rowaddr = vb + r * 128;
    const int rx = r & 7;
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      const int ch = (i & 3) * 2 + (j & 1);
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(rowaddr + (i >> 2) * 2048 + ((ch ^ rx) << 4), a0, a1, a2, a3);
      mma_bf16(s.acc[i], a0, a1, a2, a3, pb0, pb1);
    }
  }
}

// Byte offset of 16-byte chunk `ch` of row r in an FP8 tile (rows of D
// bytes; 128B swizzle for D = 128, 64B swizzle for D = 64).
template <int D>
__device__ __forceinline__ uint32_t fp8_chunk(int r, int ch) {
  if (D == 128) return r * 128 + ((ch ^ (r & 7)) << 4);
  return r * 64 + ((ch ^ ((r >> 1) & 3)) << 4);
}

// FP8 tile.
// QK on the E4M3 tensor-core MMA (m16n8k32): K fragments come straight from
// ldmatrix (row = token, 4 consecutive d bytes per register); the query is a
// two-term E4M3 split q*qs = hi + lo/16 per head (qb[2ks] = hi, qb[2ks+1] =
// lo of k-step ks), so s = s_hi + s_lo/16 keeps it to 2^-8 relative.
// PV on the f16 MMA: ldmatrix.trans of the E4M3 V rows gives each lane
// (tokens 2tq, 2tq+1) x (d 2gq, 2gq+1) of a 16-byte chunk; one byte permute
// and two exact cvt make the V^T fragments.  Output row gq of m-tile i is
// d = 16i + 2gq, row gq + 8 is d = 16i + 2gq + 1.  The per-(block, head)
// V scale multiplies the tile's P.V product in fp32.

// Masked scores (log2 units) of one FP8 tile: x = (row gq, head 2tq),
// (gq, 2tq+1), (gq+8, 2tq), (gq+8, 2tq+1).
template <int D>
__device__ __forceinline__ void qk_fp8(uint32_t kb, int valid, float4 sc,
                                       const uint32_t (&qb)[D / 16][2], float hm0,
                                       float hm1, float (&x)[4]) {
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2;
  // Four independent accumulator chains (hi/lo x even/odd k-step) keep the
  // dependent MMA depth at D/64.
  float sh[2][4] = {}, sl[2][4] = {};
  const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
  for (int ks = 0; ks < D / 32; ++ks) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(kb + fp8_chunk<D>(r, 2 * ks + (lane >> 4)), a0, a1, a2, a3);
    mma_e4m3(sh[ks & 1], a0, a1, a2, a3, qb[2 * ks][0], qb[2 * ks][1]);
    mma_e4m3(sl[ks & 1], a0, a1, a2, a3, qb[2 * ks + 1][0], qb[2 * ks + 1][1]);
  }
  // row gq is in the tile's first block, row gq + 8 in its second (bs = 8)
#pragma unroll
  for (int q = 0; q < 4; ++q)
    x[q] = fmaf(sl[0][q] + sl[1][q], 0.0625f, sh[0][q] + sh[1][q]) *
           ((q < 2 ? sc.x : sc.y) * ((q & 1) ? hm1 : hm0));
  if (gq >= valid) x[0] = x[1] = -INFINITY;
  if (gq + 8 >= valid) x[2] = x[3] = -INFINITY;
}

// O^T += vmax * (V8^T . P'^T) for one FP8 tile, P' = p * v_scale(row) / vmax.
template <int D>
__device__ __forceinline__ void pv_fp8(uint32_t vb, float vmax, uint32_t pb0,
                                       uint32_t pb1, SegState<D>& s) {
  const int lane = threadIdx.x & 31;
  const int j = lane >> 3;
  const int r = (lane & 7) + (j & 1) * 8;  // token row
#pragma unroll
  for (int pp = 0; pp < D / 32; ++pp) {
    uint32_t v0, v1, v2, v3;  // (tok 0-7, ch 2pp), (8-15, 2pp), (0-7, 2pp+1), (8-15, 2pp+1)
    ldsm_x4_t(vb + fp8_chunk<D>(r, 2 * pp + (j >> 1)), v0, v1, v2, v3);
    // [t d, t d+1, t+1 d, t+1 d+1] -> [t d, t+1 d, t d+1, t+1 d+1]
    const uint32_t u0 = __byte_perm(v0, 0, 0x3120);
    const uint32_t u1 = __byte_perm(v1, 0, 0x3120);
    const uint32_t u2 = __byte_perm(v2, 0, 0x3120);
    const uint32_t u3 = __byte_perm(v3, 0, 0x3120);
    float t0[4], t1[4];
    mma_f16_zero_c(t0, e4m3x2_to_f16x2(static_cast<uint16_t>(u0)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(u0 >> 16)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(u1)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(u1 >> 16)), pb0, pb1);
    mma_f16_zero_c(t1, e4m3x2_to_f16x2(static_cast<uint16_t>(u2)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(u2 >> 16)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(u3)),
                   e4m3x2_to_f16x2(static_cast<uint16_t>(u3 >> 16)), pb0, pb1);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      s.acc[2 * pp][q] = fmaf(vmax, t0[q], s.acc[2 * pp][q]);
      s.acc[2 * pp + 1][q] = fmaf(vmax, t1[q], s.acc[2 * pp + 1][q]);
    }
  }
}

template <int D>
__device__ __forceinline__ void tile_fp8(const DecodeParams& p, uint32_t kb,
                                         uint32_t vb, int valid, float4 sc,
                                         const uint32_t (&qb)[D / 16][2],
                                         float hm0, float hm1,
                                         SegState<D>& s) {
  float x[4];
  qk_fp8<D>(kb, valid, sc, qb, hm0, hm1, x);
  const float vmax = fmaxf(sc.z, sc.w);
  // ratios <= 1 of the two blocks' V scales (equal for block_size >= 16)
  const float r0 = __fdividef(sc.z, vmax), r1 = __fdividef(sc.w, vmax);
  float alpha0, alpha1;
  uint32_t pb0, pb1;
  softmax_tile<true>(x[0], x[1], x[2], x[3], s.m, s.l, r0, r1, alpha0, alpha1, pb0, pb1);
  rescale(s, alpha0, alpha1);
  pv_fp8<D>(vb, vmax, pb0, pb1, s);
}

// Two consecutive FP8 tiles of one segment in one step: the QK and PV
// chains of the two tiles are independent, and one conditional-max check
// (and, when needed, one cross-lane reduction) covers all 32 tokens.
template <int D>
__device__ __forceinline__ void tile_fp8_pair(uint32_t kbA, uint32_t vbA, float4 scA,
                                              uint32_t kbB, uint32_t vbB, int validB,
                                              float4 scB,
                                              const uint32_t (&qb)[D / 16][2],
                                              float hm0, float hm1, SegState<D>& s) {
  float xa[4], xb[4];
  qk_fp8<D>(kbA, kTile, scA, qb, hm0, hm1, xa);
  qk_fp8<D>(kbB, validB, scB, qb, hm0, hm1, xb);
  constexpr float kSlack = 8.f;  // as in softmax_tile
  const float t0 = fmaxf(fmaxf(xa[0], xa[2]), fmaxf(xb[0], xb[2]));
  const float t1 = fmaxf(fmaxf(xa[1], xa[3]), fmaxf(xb[1], xb[3]));
  float alpha0 = 1.f, alpha1 = 1.f;
  if (__any_sync(0xffffffffu, t0 > s.m[0] + kSlack || t1 > s.m[1] + kSlack)) {
    float mx0 = t0, mx1 = t1;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(s.m[0], mx0), mn1 = fmaxf(s.m[1], mx1);
    alpha0 = fast_exp2(s.m[0] - mn0);
    alpha1 = fast_exp2(s.m[1] - mn1);
    s.m[0] = mn0;
    s.m[1] = mn1;
  }
  float pa[4], pb[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    pa[q] = fast_exp2(xa[q] - s.m[q & 1]);
    pb[q] = fast_exp2(xb[q] - s.m[q & 1]);
  }
  s.l[0] = s.l[0] * alpha0 + ((pa[0] + pa[2]) + (pb[0] + pb[2]));
  s.l[1] = s.l[1] * alpha1 + ((pa[1] + pa[3]) + (pb[1] + pb[3]));
  const float vmaxA = fmaxf(scA.z, scA.w), vmaxB = fmaxf(scB.z, scB.w);
  const float ra0 = __fdividef(scA.z, vmaxA), ra1 = __fdividef(scA.w, vmaxA);
  const float rb0 = __fdividef(scB.z, vmaxB), rb1 = __fdividef(scB.w, vmaxB);
  const uint32_t pbA0 = movmatrix_t(pack_f16x2(pa[0] * ra0, pa[1] * ra0));
  const uint32_t pbA1 = movmatrix_t(pack_f16x2(pa[2] * ra1, pa[3] * ra1));
  const uint32_t pbB0 = movmatrix_t(pack_f16x2(pb[0] * rb0, pb[1] * rb0));
  const uint32_t pbB1 = movmatrix_t(pack_f16x2(pb[2] * rb1, pb[3] * rb1));
  rescale(s, alpha0, alpha1);
  pv_fp8<D>(vbA, vmaxA, pbA0, pbA1, s);
  pv_fp8<D>(vbB, vmaxB, pbB0, pbB1, s);
}

// d index of accumulator element (i, q) for lane gq.
template <int D, bool FP8>
__device__ __forceinline__ int acc_d(int i, int q, int gq) {
  if (!FP8) return 16 * i + gq + ((q >> 1) << 3);
  // FP8: m-tile i covers chunk i; rows gq / gq + 8 are d = 16i + 2gq (+1).
  return 16 * i + 2 * gq + (q >> 1);
}

template <int D, bool FP8>
__device__ __forceinline__ void consumer(const DecodeParams& p, Header* hdr,
                                         uint32_t qbuf, uint32_t ring,
                                         int64_t lo, int64_t hi,
                                         int32_t cta) {
  using L = Smem<D, FP8>;
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  Cursor c;
  locate(p, lo, c);
  int64_t u = lo;
  uint32_t it = 0, qcount = 0;
  bool ok = true;
  SegState<D> s;
  uint32_t qb[D / 16][2];
  while (u < hi && ok) {
    const int32_t seg_end = static_cast<int32_t>(
        min(static_cast<int64_t>(c.T), c.tile + (hi - u)));
    const bool whole = c.tile == 0 && seg_end == c.T;
    // ---- query fragments (B operand, n = head, k = d)
    const uint32_t qslot = qbuf + (qcount & 1) * L::kQBytes;
    ok = mbar_wait(smem_addr(&hdr->qfull[qcount & 1]), (qcount >> 1) & 1);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    float hm0 = p.scale_log2, hm1 = p.scale_log2;
    if (!FP8) {
#pragma unroll
      for (int kp = 0; kp < D / 32; ++kp) {
        const int kk = 2 * kp;
        const int r = lane & 7;
        const int ch = (kk & 3) * 2 + (lane >> 3);
        ldsm_x4(qslot + (kk >> 2) * L::kQSlabBytes + r * 128 + ((ch ^ r) << 4),
                qb[kk][0], qb[kk][1], qb[kk + 1][0], qb[kk + 1][1]);
      }
    } else {
      // q[gq][32ks + 16h + 4tq .. +3] (h = 0, 1) as a two-term E4M3 split
      // per head: x = q * qs with the power of two qs putting max|x| in
      // [128, 256); hi = e4m3(x), lo = e4m3(16 (x - hi)); B fragments
      // qb[2ks][h] = hi, qb[2ks + 1][h] = lo.  The scores are divided by qs.
      float qv[D / 32][2][4];
      float amax = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 32; ++ks)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int byte = (32 * ks + 16 * h + 4 * tq) * 2;  // within the row
          const int slab = byte >> 7, inrow = byte & 127;
          const int ch = inrow >> 4;
          const uint32_t addr = qslot + slab * L::kQSlabBytes + gq * 128 +
                                ((ch ^ gq) << 4) + (inrow & 15);
          uint32_t w0, w1;
          asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];"
                       : "=r"(w0), "=r"(w1)
                       : "r"(addr)
                       : "memory");
          const float2 f0 = unpack_bf16x2(w0), f1 = unpack_bf16x2(w1);
          qv[ks][h][0] = f0.x; qv[ks][h][1] = f0.y; qv[ks][h][2] = f1.x; qv[ks][h][3] = f1.y;
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)),
                                   fmaxf(fabsf(f1.x), fabsf(f1.y))));
        }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      // amax in [2^(e-1), 2^e) from the exponent field (subnormal or zero
      // amax clamps to e = -100, which keeps every power of two below normal)
      int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 126;
      e = max(e, -100);
      const float qs = __uint_as_float(static_cast<uint32_t>(8 - e + 127) << 23);
#pragma unroll
      for (int ks = 0; ks < D / 32; ++ks)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float x[4], r[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) x[k] = qv[ks][h][k] * qs;
          const uint32_t h01 = f32x2_to_e4m3x2(x[0], x[1]);
          const uint32_t h23 = f32x2_to_e4m3x2(x[2], x[3]);
          const float2 d01 = unpack_f16x2(e4m3x2_to_f16x2(static_cast<uint16_t>(h01)));
          const float2 d23 = unpack_f16x2(e4m3x2_to_f16x2(static_cast<uint16_t>(h23)));
          r[0] = (x[0] - d01.x) * 16.f;
          r[1] = (x[1] - d01.y) * 16.f;
          r[2] = (x[2] - d23.x) * 16.f;
          r[3] = (x[3] - d23.y) * 16.f;
          qb[2 * ks][h] = h01 | (h23 << 16);
          qb[2 * ks + 1][h] = f32x2_to_e4m3x2(r[0], r[1]) | (f32x2_to_e4m3x2(r[2], r[3]) << 16);
        }
      const float inv = p.scale_log2 * __uint_as_float(static_cast<uint32_t>(e - 8 + 127) << 23);
      hm0 = __shfl_sync(0xffffffffu, inv, (2 * tq) * 4);
      hm1 = __shfl_sync(0xffffffffu, inv, (2 * tq + 1) * 4);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&hdr->qempty[qcount & 1]));
    ++qcount;
    seg_reset(s);
    // ---- tiles
    for (int32_t tile = c.tile; tile < seg_end; ++tile) {
      if (FP8 && tile + 1 < seg_end) {
        // Two full-or-tail tiles in one step (the first is never a tail).
        const uint32_t sA = it % p.stages, sB = (it + 1) % p.stages;
        ok = mbar_wait(smem_addr(&hdr->full[sA]), (it / p.stages) & 1);
        ok = ok && mbar_wait(smem_addr(&hdr->full[sB]), ((it + 1) / p.stages) & 1);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint32_t kbA = ring + sA * L::kStageBytes, kbB = ring + sB * L::kStageBytes;
        const int validB = min(kTile, c.n - (tile + 1) * kTile);
        if (validB < kTile) {
          for (int off = validB * D + lane * 16; off < kTile * D; off += 32 * 16)
            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(kbB + L::kKVBytes + off), "r"(0)
                         : "memory");
          fence_proxy_async_smem();
          __syncwarp();
        }
        tile_fp8_pair<D>(kbA, kbA + L::kKVBytes, hdr->scales[sA], kbB, kbB + L::kKVBytes,
                         validB, hdr->scales[sB], qb, hm0, hm1, s);
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_addr(&hdr->empty[sA]));
          mbar_arrive(smem_addr(&hdr->empty[sB]));
        }
        it += 2;
        ++tile;
        continue;
      }
      const uint32_t stage = it % p.stages;
      ok = mbar_wait(smem_addr(&hdr->full[stage]), (it / p.stages) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const uint32_t kb = ring + stage * L::kStageBytes;
      const uint32_t vb = kb + L::kKVBytes;
      const int valid = min(kTile, c.n - tile * kTile);
      if (valid < kTile) {
        // Rows past the sequence end hold stale or foreign data: zero the V
        // rows (0 * NaN would poison the MMA); K rows are masked by -inf.
        const int row_bytes = FP8 ? D : 128;
        for (int sl = 0; sl < L::kSlabs; ++sl)
          for (int off = valid * row_bytes + lane * 16; off < kTile * row_bytes; off += 32 * 16)
            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(vb + sl * L::kSlabBytes + off), "r"(0)
                         : "memory");
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (!FP8) {
        tile_bf16<D>(p, kb, vb, valid, qb, s);
      } else {
        tile_fp8<D>(p, kb, vb, valid, hdr->scales[stage], qb, hm0, hm1, s);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&hdr->empty[stage]));
      ++it;
    }
    if (!ok) break;
    // ---- finalise the piece
    float l0 = s.l[0], l1 = s.l[1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    const int h0 = 2 * tq, h1 = 2 * tq + 1;
    if (whole) {
      const float i0 = 1.f / l0, i1 = 1.f / l1;
      __nv_bfloat16* ob = p.out + (static_cast<int64_t>(c.b) * p.num_q_heads +
                                   c.g * p.group) * D;
#pragma unroll
      for (int i = 0; i < D / 16; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int h = (q & 1) ? h1 : h0;
          if (h < p.group)
            ob[h * D + acc_d<D, FP8>(i, q, gq)] =
                __float2bfloat16_rn(s.acc[i][q] * ((q & 1) ? i1 : i0));
        }
    } else {
      const int64_t piece = static_cast<int64_t>(cta) + c.b * p.num_kv_heads + c.g;
      float* wo = p.ws_o + piece * kMaxG * D;
#pragma unroll
      for (int i = 0; i < D / 16; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int h = (q & 1) ? h1 : h0;
          if (h < p.group) wo[h * D + acc_d<D, FP8>(i, q, gq)] = s.acc[i][q];
        }
      if (gq == 0) {
        if (h0 < p.group) p.ws_ml[piece * kMaxG + h0] = make_float2(s.m[0], l0);
        if (h1 < p.group) p.ws_ml[piece * kMaxG + h1] = make_float2(s.m[1], l1);
      }
    }
    u += seg_end - c.tile;
    if (u < hi) next_segment(p, c);
  }
}

template <int D, bool FP8>
__global__ void __launch_bounds__(64)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const DecodeParams p) {
  using L = Smem<D, FP8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Header* hdr = reinterpret_cast<Header*>(smem_raw);
  const uint32_t base = smem_addr(smem_raw);
  // Swizzled TMA boxes need 1024-byte aligned destinations; the dynamic
  // shared window is expected to start aligned.  Check rather than assume.
  if (base & 1023u) {
    if (threadIdx.x == 0) flag_error(PA_DEVERR_LAUNCH);
    return;
  }
  const uint32_t tiles = base + L::kHeaderBytes;
  const uint32_t qbuf = tiles;
  const uint32_t ring = tiles + 2 * L::kQBytes;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_addr(&hdr->full[s]), 1);
      mbar_init(smem_addr(&hdr->empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&hdr->qfull[s]), 1);
      mbar_init(smem_addr(&hdr->qempty[s]), 1);
    }
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncthreads();

  int64_t W = total_tiles(p);  // both warps compute it; identical
  if (W == 0) return;
  // With fewer tiles than CTAs only the first W CTAs take part, so that
  // every participating CTA owns at least one tile (the merge relies on it).
  const int32_t P = static_cast<int32_t>(min(static_cast<int64_t>(p.num_ctas), W));
  if (static_cast<int32_t>(blockIdx.x) >= P) return;
  int64_t lo, hi;
  cta_range(W, P, blockIdx.x, lo, hi);
  if (warp == 0)
    producer<D, FP8>(p, &tm_q, &tm_k, &tm_v, hdr, qbuf, ring, lo, hi);
  else
    consumer<D, FP8>(p, hdr, qbuf, ring, lo, hi, blockIdx.x);
  (void)lane;
}

// ----------------------------------------------------------------- merge --
// One CTA per segment (b, g).  Empty sequences get zeros; segments covered
// by a single CTA were written by the decode kernel; split segments combine
// their pieces:  M = max_j m_j,  out = sum_j 2^(m_j - M) o_j /
// sum_j 2^(m_j - M) l_j.
template <int D>
__global__ void __launch_bounds__(256)
    paged_decode_merge_kernel(const DecodeParams p) {
  const int32_t seg = blockIdx.x;
  const int32_t b = seg / p.num_kv_heads, g = seg % p.num_kv_heads;
  __shared__ int64_t s_before;
  __shared__ int64_t s_W;
  const int32_t n = clamp_len(p, p.seq_lens[b]);
  const int32_t T = cdiv16(n);
  __nv_bfloat16* ob = p.out + (static_cast<int64_t>(b) * p.num_q_heads + g * p.group) * D;
  if (T == 0) {
    for (int i = threadIdx.x; i < p.group * D; i += blockDim.x)
      ob[i] = __float2bfloat16_rn(0.f);
    return;
  }
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int64_t before = 0, all = 0;
    for (int32_t bb = lane; bb < p.num_seqs; bb += 32) {
      const int64_t t = cdiv16(clamp_len(p, p.seq_lens[bb]));
      all += t;
      if (bb < b) before += t;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      all += __shfl_xor_sync(0xffffffffu, all, o);
    }
    if (lane == 0) {
      s_before = before * p.num_kv_heads;
      s_W = all * p.num_kv_heads;
    }
  }
  __syncthreads();
  const int64_t start = s_before + static_cast<int64_t>(g) * T;
  const int64_t W = s_W;
  const int32_t P = static_cast<int32_t>(min(static_cast<int64_t>(p.num_ctas), W));
  const int32_t c0 = cta_of(W, P, start);
  const int32_t c1 = cta_of(W, P, start + T - 1);
  if (c0 == c1) return;
  const int64_t pbase = static_cast<int64_t>(seg);
  for (int idx = threadIdx.x; idx < p.group * D; idx += blockDim.x) {
    const int h = idx / D;
    float M = -INFINITY;
    for (int32_t c = c0; c <= c1; ++c)
      M = fmaxf(M, p.ws_ml[(pbase + c) * kMaxG + h].x);
    float num = 0.f, den = 0.f;
    for (int32_t c = c0; c <= c1; ++c) {
      const float2 ml = p.ws_ml[(pbase + c) * kMaxG + h];
      const float w = fast_exp2(ml.x - M);
      num = fmaf(w, p.ws_o[(pbase + c) * kMaxG * D + idx], num);
      den = fmaf(w, ml.y, den);
    }
    ob[idx] = __float2bfloat16_rn(num / den);
  }
}

}  // namespace pa
