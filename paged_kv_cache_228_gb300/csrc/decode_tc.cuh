// Paged single-token decode over an FP8 (E4M3) cache on the fifth-generation
// tensor cores (tcgen05 UMMA, kind::f8f6f4), head_dim 128.
//
// Method: the same result as the other decode kernels -- dense attention
// over each request's logical sequence, gathered through its block table
// ("Paged Attention and KV Cache Fragmentation", section "How PagedAttention
// maps an OS concept onto GPU memory"; "KV cache fragmentation" (field
// guide), section "Definition") -- over a cache whose per-(block, head)
// scales are applied in fp32 and whose products accumulate in fp32
// ("Paged Attention and KV Cache Fragmentation", section "Quantization as a
// way to stretch paged memory further").
//
// GB300 design
// ------------
// * Work: the cost-weighted split of the flat 16-token tile list that every
//   decode kernel uses (my_range), taken in chunks of up to 16 tiles of one
//   (sequence, KV head) segment: 256 tokens, two M = 128 QK MMAs per K step
//   and a K = 256 PV.  Each softmax thread takes two tokens of a chunk, so
//   the per-chunk waits and barriers are shared by twice the data (128-token
//   chunks measured 377 us against 329 at 128K).
// * A CTA (one per SM) is 14 warps with fixed roles:
//     warps 0, 11-13  copies: each chunk's K and V boxes by TMA into a ring
//                stage (K by two warps, V by two: one warp's TMA issue is
//                too slow for the chunk rate), its blocks' scales by
//                cp.async (both complete on the stage's barrier), each
//                piece's query rows by TMA;
//     warp 1     splits the piece's query per head into two E4M3 terms,
//                x = q * 2^s = hi + lo / 16, as the 16 rows of the B
//                operand, then per chunk the QK MMAs
//                  S^T[2 x 128 tok x 16] = K[256 x 128 d] . [hi; lo]^T;
//     warp 10    per chunk, once its P is written, the PV MMAs
//                  O^T[128 d x 16]   = V^T[128 d x 256 tok] . [P_hi; P_lo]^T
//                (two issuing warps, so the next chunk's QK never delays
//                this chunk's PV), both into tensor memory (fp32);
//     warps 2-9  two groups of four (one warp per tensor-memory lane
//                quarter), group g taking heads 4g .. 4g + 3: two tokens
//                per thread (t and t + 128), the score s = (S_hi + S_lo / 16) * k_scale *
//                scale / 2^s, the online softmax, P written to shared
//                memory as a two-term E4M3 split; then, as d = lane of the
//                same quarter, the chunk's O^T added into fp32 registers,
//                and at a piece's end its output.
// * The running max of a head is shared by the 256 tokens of a chunk and
//   moves only when a score passes it by more than kTcSlack (log2 units):
//   one barrier reduction per chunk decides that for each group.  So P <= 2^kTcSlack.
// * V scales: P' = p * v_scale(block) / vmax(chunk) * kTcPScale <= 256, and
//   the chunk's O^T is in units of vmax(chunk) / kTcPScale, applied when it
//   is added to the registers.  The two-term split keeps P' to 2^-8
//   relative (absolute 2^-14 where the lo term is subnormal); a bf16 query
//   it carries exactly above about 2^-14 of its row's largest element.
// * Shared memory: [ring stages of K | V (32 KB each) | 2 query slots (bf16)
//   | 2 E4M3 query operands | 2 P buffers | header].  K tiles are K-major
//   and V tiles MN-major operands with the 128-byte swizzle the TMA writes;
//   P is an MN-major operand without swizzle.
#pragma once

#include "decode.cuh"
#include "umma.cuh"

namespace pa {

// Every wait of this kernel: at most kTcSuspendNs per poll (the phase's
// completion ends it earlier), so waiting warps leave the issue slots to
// the others; p.wait_limit (default) polls bound it to about 8 s.
constexpr uint32_t kTcSuspendNs = 2000;
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity,
                                        uint32_t limit = (1u << 22)) {
  return mbar_wait_sleep(bar, parity, limit, kTcSuspendNs);
}

constexpr int kTcTiles = 16;              // 16-token tiles per chunk
constexpr int kTcTok = kTcTiles * kTile;  // tokens per chunk
constexpr int kTcM = 128;                 // tokens per QK MMA (its M)
constexpr int kTcHalves = kTcTok / kTcM;  // QK MMAs per K step; tokens per softmax thread
constexpr int kTcMaxStages = 6;
constexpr int kTcCopyWarps = 4;  // K and V boxes split over these (even)
constexpr int kTcSoftWarps = 8;  // two per tensor-memory lane quarter
constexpr int kTcGroupHeads = 4; // heads per softmax warp (group of four warps)
constexpr int kTcThreads = 32 * (2 + kTcSoftWarps + kTcCopyWarps);
constexpr float kTcSlack = 4.f;    // log2 units the max may lag the scores
constexpr float kTcPScale = 16.f;  // 2^(8 - kTcSlack): P' <= 256 < 448
// tensor memory: S of chunk parity b at columns kTcSCols b (+ 16 per half),
// O at kTcOCol + 16 b
constexpr uint32_t kTcSCols = 16 * kTcHalves;
constexpr uint32_t kTcOCol = 2 * kTcSCols;
constexpr uint32_t kTcTmemCols = 128;
static_assert(kTcOCol + 32 <= kTcTmemCols, "tensor memory columns");
// Named barriers 1 and 2: the four softmax warps of group 0, resp. 1 (as
// constants, so the kernel reserves only the barriers it names).
__device__ __forceinline__ void tc_group_sync(int g) {
  if (g == 0)
    named_bar_sync<1>(128);
  else
    named_bar_sync<2>(128);
}
__device__ __forceinline__ uint32_t tc_group_popc(int g, bool pred) {
  return g == 0 ? named_bar_popc<1>(128, pred) : named_bar_popc<2>(128, pred);
}

template <int D>
struct TcSmem {
  static constexpr int kKV = kTcTok * D;           // K (or V) of one chunk
  static constexpr int kStage = 2 * kKV;
  static constexpr int kQ = kMaxG * D * 2;         // bf16 query rows, D/64 slabs
  static constexpr int kQ8 = 2 * kMaxG * D;        // [hi; lo] rows of D bytes
  static constexpr int kP = kTcTok * 2 * kMaxG;    // 16 bytes per token
};

struct TcHeader {
  uint64_t full[kTcMaxStages];   // chunk landed (TMA bytes, scale copies, arrive)
  uint64_t empty[kTcMaxStages];  // chunk's MMAs done
  uint64_t qfull[2], qempty[2];  // bf16 query slot landed / split
  uint64_t qready[2];            // E4M3 query operand and hm written
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2];
  uint64_t o_full[2], o_empty[2];
  uint64_t mma_done[2];           // each issuing warp's MMAs complete
  uint64_t stall;                 // test hook: never arrived at
  float sk[kTcMaxStages][32];     // K scale per box (8 or 16 tokens)
  float sv[kTcMaxStages][32];     // V scale per box
  int32_t ent[kTcCopyWarps][4][32];  // copy part w, lane l: entry of chunk c at [w][c & 3][l]
  float hm[2][kMaxG];             // per head: scale * log2(e) / 2^s
  float red_m[2][4][kTcGroupHeads];     // group, warp quarter: chunk maxima
  float red_l[2][2][4][kTcGroupHeads];  // parity, group, quarter: sums at a piece's end
  alignas(16) float red_v[2][2][4];     // parity, group, quarter: largest V scale
  uint32_t tmem;
};

template <int D>
__host__ __device__ constexpr size_t tc_smem_bytes(int stages) {
  using L = TcSmem<D>;
  return static_cast<size_t>(stages) * L::kStage + 2 * L::kQ + 2 * L::kQ8 + 2 * L::kP +
         sizeof(TcHeader);
}

// ------------------------------------------------------------ chunking ---
// The work split runs in whole chunks (tile_log2 = log2 kTcTiles: a
// segment is ceil(n / 256) work units), so a CTA's range never cuts a chunk
// and every chunk but a segment's last is full: a chunk costs about the
// same whatever its number of tokens.  A chunk: the kTcTiles tiles of one
// work unit of a segment (fewer at the sequence's end).  Every role walks
// the same sequence of chunks.
struct TcIter {
  Cursor c;         // segment; c.tile, c.T in chunks
  int64_t u;        // flat index of the chunk
  int64_t useg;     // flat index of the segment's chunk 0
  int32_t seg_end;  // end of this CTA's part (piece) of the segment, in chunks
  int32_t nt;       // 16-token tiles in the chunk; 0 past the range
  bool first;       // the chunk opens the piece
  bool whole;       // the piece is the whole segment
};

// 16-token tiles of chunk c.tile of the sequence.
__device__ __forceinline__ int32_t tc_chunk_tiles(const Cursor& c) {
  return min(kTcTiles, cdiv16(c.n) - c.tile * kTcTiles);
}

__device__ __forceinline__ void tc_open_piece(TcIter& it, int64_t hi) {
  it.seg_end = static_cast<int32_t>(min(static_cast<int64_t>(it.c.T), it.c.tile + (hi - it.u)));
  it.useg = it.u - it.c.tile;
  it.whole = it.c.tile == 0 && it.seg_end == it.c.T;
  it.first = true;
  it.nt = tc_chunk_tiles(it.c);
}

__device__ __forceinline__ void tc_next(const DecodeParams& p, TcIter& it, int64_t hi) {
  if (it.nt == 0) return;
  ++it.u;
  ++it.c.tile;
  if (it.c.tile < it.seg_end) {
    it.first = false;
    it.nt = tc_chunk_tiles(it.c);
    return;
  }
  if (it.u >= hi) {
    it.nt = 0;
    return;
  }
  next_segment(p, it.c);
  tc_open_piece(it, hi);
}

__device__ __forceinline__ bool tc_last(const TcIter& it) { return it.c.tile + 1 == it.seg_end; }

// Tokens of the chunk inside the sequence (>= 1).
__device__ __forceinline__ int32_t tc_valid(const TcIter& it) {
  return min(it.nt * kTile, it.c.n - it.c.tile * kTcTok);
}

// --------------------------------------------------------------- copies ---
// Lane l's box of the chunk (box = block_size rows for block_size 8, else
// 16 rows) into entry slot `dst` of shared memory: its block-table entry by
// cp.async, or -2 when the box is past the chunk or the sequence.
__device__ __forceinline__ void tc_fetch_entry(const DecodeParams& p, const TcIter& it, int lr,
                                               uint32_t dst) {
  const int lane = threadIdx.x & 31;
  const int32_t t = lane >> lr;
  const int32_t tok = (it.c.tile * kTcTiles + t) * kTile + (lane & ((1 << lr) - 1)) * p.block_size;
  if (it.nt == 0 || t >= it.nt || tok >= it.c.n) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(dst), "r"(-2) : "memory");
    return;
  }
  cp_async4(dst, p.block_tables + static_cast<int64_t>(it.c.b) * p.max_blocks + (tok >> p.log2_bs));
}

// Copy warps: part p of kTcCopyWarps issues the chunk's K (p even) or V (p
// odd) boxes b with b % (kTcCopyWarps / 2) == p / 2 -- one warp's TMA issue
// alone is too slow for the chunk rate; part 0 also copies the scales and a
// new piece's query rows.  Each fetches the chunk's
// block-table entries two chunks ahead by cp.async into its own shared slots
// (the copy group of two chunks back is waited for, so no register ever
// waits on a load), and issues a chunk as soon as its stage is free.
// Returns after every copy it issued has landed.
template <int D>
__device__ __forceinline__ void tc_produce(const DecodeParams& p, const CUtensorMap* tq,
                                           const CUtensorMap* tkv, int part, uint32_t ring,
                                           uint32_t qbuf, TcHeader* hdr, TcIter it0, int64_t hi) {
  using L = TcSmem<D>;
  const int lane = threadIdx.x & 31;
  const int lr = p.block_size < kTile ? 1 : 0;
  const int box_rows = p.block_size < kTile ? p.block_size : kTile;
  const uint32_t box_bytes = static_cast<uint32_t>(box_rows) * D;
  const uint32_t S = p.stages;
  const uint32_t ent = smem_addr(&hdr->ent[part][0][lane]);  // slot c & 3 at + (c & 3) * 128
  const int kv = part & 1;
  const bool mine = (lane % (kTcCopyWarps / 2)) == (part >> 1);  // this warp's boxes
  TcIter it1 = it0;
  tc_next(p, it1, hi);
  TcIter it2 = it1;
  tc_next(p, it2, hi);
  tc_fetch_entry(p, it0, lr, ent);
  cp_async_commit();
  tc_fetch_entry(p, it1, lr, ent + 128);
  cp_async_commit();
  uint32_t j = 0, qn = 0, st = 0, ph = 0;  // chunk, query slots used, stage, its use
  for (; it0.nt > 0; ++j) {
    bool ok = true;
    if (lane == 0) {
      if (j >= S) ok = tc_wait(smem_addr(&hdr->empty[st]), ph ^ 1);
      if (ok && part == 0 && it0.first && qn >= 2)
        ok = tc_wait(smem_addr(&hdr->qempty[qn & 1]), ((qn >> 1) - 1) & 1);
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    cp_async_wait_group<1>();  // this chunk's entries (two groups back) landed
    int32_t e;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(e) : "r"(ent + (j & 3) * 128) : "memory");
    if (part == 0 && it0.first) {
      if (lane == 0) {
        const uint32_t bar = smem_addr(&hdr->qfull[qn & 1]);
        mbar_arrive_expect_tx(bar, L::kQ);
        const int32_t row = it0.c.b * p.num_q_heads + it0.c.g * p.group;
#pragma unroll
        for (int sl = 0; sl < D / 64; ++sl)
          tma_load_2d(qbuf + (qn & 1) * L::kQ + sl * 1024, tq, sl * 64, row, bar);
      }
      ++qn;
    }
    const uint32_t full = smem_addr(&hdr->full[st]);
    const bool has = e != -2;
    const bool good = has && e >= 0 && e < p.num_blocks;
    const uint32_t nbox = __popc(__ballot_sync(0xffffffffu, has && mine));
    if (lane == 0) mbar_expect_tx(full, nbox * box_bytes);
    __syncwarp();
    if (has && (mine || part == 0)) {
      int32_t row;
      if (good) {
        const int32_t tok = (it0.c.tile * kTcTiles + (lane >> lr)) * kTile;
        row = (e * p.num_kv_heads + it0.c.g) * p.block_size + (lr ? 0 : (tok & (p.block_size - 1)));
      } else {
        if (mine) flag_error(PA_DEVERR_BAD_BLOCK_ID);
        row = p.rows_total;  // out of the tensor: zero fill
      }
      if (mine) tma_load_2d(ring + st * L::kStage + kv * L::kKV + lane * box_bytes, tkv, 0, row, full);
      const uint32_t sk = smem_addr(&hdr->sk[st][lane]), sv = smem_addr(&hdr->sv[st][lane]);
      if (part != 0) {
      } else if (good) {
        const int64_t x = static_cast<int64_t>(e) * p.num_kv_heads + it0.c.g;
        cp_async4(sk, p.k_scale + x);
        cp_async4(sv, p.v_scale + x);
      } else {
        st_shared_f32(sk, 1.f);
        st_shared_f32(sv, 1.f);
      }
    }
    if (part == 0) cp_async_mbar_arrive(full);  // the scales above complete the stage too
    tc_fetch_entry(p, it2, lr, ent + ((j + 2) & 3) * 128);
    cp_async_commit();
    __syncwarp();
    if (lane == 0) mbar_arrive(full);
    it0 = it1;
    it1 = it2;
    tc_next(p, it2, hi);
    if (++st == S) {
      st = 0;
      ph ^= 1;
    }
  }
  cp_async_wait_group<0>();
  // No copy may still target shared memory when the CTA exits.
  if (lane == 0) {
    for (uint32_t k = j > S ? j - S : 0; k < j; ++k)
      tc_wait(smem_addr(&hdr->full[k % S]), (k / S) & 1, 1u << 16);
    for (uint32_t k = qn > 2 ? qn - 2 : 0; k < qn; ++k)
      tc_wait(smem_addr(&hdr->qfull[k & 1]), (k >> 1) & 1, 1u << 16);
  }
  __syncwarp();
}

// -------------------------------------------------------- tensor cores ---
// Two non-negative or signed values below 448 in magnitude -> their
// two-term E4M3 split hi = e4m3(x), lo = e4m3(16 (x - hi)) through f16 (x
// rounded to f16 first; 16 (x - hi) is exact there).  First value in the
// low byte.
__device__ __forceinline__ void split_e4m3x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 x = __floats2half2_rn(a, b);
  const __nv_fp8x2_storage_t h =
      __nv_cvt_halfraw2_to_fp8x2(static_cast<__half2_raw>(x), __NV_SATFINITE, __NV_E4M3);
  const __half2 xh = __half2(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3));
  const __half2 r = __hfma2(xh, __float2half2_rn(-16.f), __hmul2(x, __float2half2_rn(16.f)));
  const __nv_fp8x2_storage_t l =
      __nv_cvt_halfraw2_to_fp8x2(static_cast<__half2_raw>(r), __NV_SATFINITE, __NV_E4M3);
  hi = h;
  lo = l;
}

// Operand row (= column of S and O) of head h's hi term; its lo term is 4
// rows further.  Heads 4g .. 4g + 3 and their two terms are the 8
// consecutive columns 8g .. 8g + 7 that softmax group g reads.
__device__ __forceinline__ int tc_col(int h) { return 8 * (h >> 2) + (h & 3); }

// Warp 1: the query rows of a segment (bf16 slot as the TMA wrote it) ->
// the E4M3 B operand rows (hi and lo of every head, at tc_col), K-major,
// 128-byte swizzle, and hm[h] = scale * log2(e) / 2^s_h.  Lane (h = lane / 4, part =
// lane % 4) takes d = 32 part .. 32 part + 31 of head h; the power of two
// 2^s_h puts max |q_h| * 2^s_h in [128, 256).  Heads past the group give
// zero rows.
template <int D>
__device__ __forceinline__ void tc_split_query(const DecodeParams& p, uint32_t qslot,
                                               uint32_t q8, float* hm) {
  static_assert(D == 128, "one lane quarter per 32 values of d");
  const int lane = threadIdx.x & 31;
  const int h = lane >> 2, part = lane & 3;
  float v[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int ch = (part & 1) * 4 + i;
    uint32_t w[4];
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(qslot + (part >> 1) * 1024 + h * 128 + ((ch ^ h) << 4))
                 : "memory");
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = unpack_bf16x2(w[k]);
      v[8 * i + 2 * k] = f.x;
      v[8 * i + 2 * k + 1] = f.y;
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  // amax in [2^(e-1), 2^e) from its exponent field (zero or subnormal
  // clamps to e = -100, which keeps both powers of two normal)
  int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 126;
  e = max(e, -100);
  const float qs = __uint_as_float(static_cast<uint32_t>(8 - e + 127) << 23);
  const bool live = h < p.group;
  uint32_t hw[8], lw[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint32_t h0, l0, h1, l1;
    split_e4m3x2(v[4 * k] * qs, v[4 * k + 1] * qs, h0, l0);
    split_e4m3x2(v[4 * k + 2] * qs, v[4 * k + 3] * qs, h1, l1);
    hw[k] = live ? (h0 | (h1 << 16)) : 0u;
    lw[k] = live ? (l0 | (l1 << 16)) : 0u;
  }
  const int rh = tc_col(h), rl = rh + 4;  // rows of the two terms
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int ch = 2 * part + cc;
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(q8 + rh * 128 + ((ch ^ (rh & 7)) << 4)),
                 "r"(hw[4 * cc]), "r"(hw[4 * cc + 1]), "r"(hw[4 * cc + 2]), "r"(hw[4 * cc + 3])
                 : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(q8 + rl * 128 + ((ch ^ (rl & 7)) << 4)),
                 "r"(lw[4 * cc]), "r"(lw[4 * cc + 1]), "r"(lw[4 * cc + 2]), "r"(lw[4 * cc + 3])
                 : "memory");
  }
  if (part == 0)
    hm[h] = live ? p.scale_log2 * __uint_as_float(static_cast<uint32_t>(e - 8 + 127) << 23) : 0.f;
}

// Warp 1: for every chunk in order, once its stage has landed and its S
// buffer is free, the QK MMAs (after splitting the query of a new piece).
// Waits are bounded (p.wait_limit polls); on a timeout the warp stops.
template <int D>
__device__ __forceinline__ void tc_mma_qk(const DecodeParams& p, uint32_t ring, uint32_t qbuf,
                                          uint32_t q8buf, TcHeader* hdr, uint32_t tmem,
                                          TcIter it, int64_t hi) {
  using L = TcSmem<D>;
  const int lane = threadIdx.x & 31;
  const uint32_t S = p.stages, wl = p.wait_limit;
  constexpr uint32_t kIdQK = idesc_e4m3(kTcM, 2 * kMaxG, false, false);
  // descriptors of stage 0 and query slot 0; other buffers and every K step
  // add their byte offset >> 4 to the start-address field (shared addresses
  // are below 256 KB, so the field never carries)
  const uint64_t kd0 = smem_desc(ring, 16, 1024, 2);
  const uint64_t qd0 = smem_desc(q8buf, 16, 1024, 2);
  uint64_t qd = qd0;
  uint32_t sg = 0;
  for (uint32_t j = 0; it.nt > 0; ++j) {
    const uint32_t st = j % S;
    bool ok = tc_wait(smem_addr(&hdr->full[st]), (j / S) & 1, wl);
    // (s_empty also means the softmax warps have read hm of the piece that
    // last used this query slot)
    if (ok && j >= 2) ok = tc_wait(smem_addr(&hdr->s_empty[j & 1]), ((j >> 1) - 1) & 1, wl);
    if (ok && it.first) ok = tc_wait(smem_addr(&hdr->qfull[sg & 1]), (sg >> 1) & 1, wl);
    if (!__all_sync(0xffffffffu, ok)) break;
    if (it.first) {
      const uint32_t slot = sg & 1;
      qd = qd0 + (slot * L::kQ8 >> 4);
      tc_split_query<D>(p, qbuf + slot * L::kQ, q8buf + slot * L::kQ8, hdr->hm[slot]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&hdr->qempty[slot]));
        mbar_arrive(smem_addr(&hdr->qready[slot]));
      }
      ++sg;
    }
    tc_fence_after_sync();
    if (lane == 0) {
      const uint64_t kd = kd0 + (st * L::kStage >> 4);
      const uint32_t ts = tmem + (j & 1) * kTcSCols;
#pragma unroll
      for (int h = 0; h < kTcHalves; ++h)
#pragma unroll
        for (int k = 0; k < D / 32; ++k)
          umma_e4m3(ts + 16 * h, kd + h * (kTcM * D >> 4) + 2 * k, qd + 2 * k, kIdQK, k > 0);
      umma_commit(smem_addr(&hdr->s_full[j & 1]));
    }
    __syncwarp();
    tc_next(p, it, hi);
  }
  // every MMA this thread issued has completed before the tensor memory is
  // released
  if (lane == 0) {
    umma_commit(smem_addr(&hdr->mma_done[0]));
    tc_wait(smem_addr(&hdr->mma_done[0]), 0, wl);
  }
  __syncwarp();
}

// Warp 6: for every chunk in order, once its P is written and its O buffer
// is free, the PV MMAs; their completion frees the chunk's stage.  A second
// issuing warp keeps the QK MMAs of the next chunk from delaying them.
template <int D>
__device__ __forceinline__ void tc_mma_pv(const DecodeParams& p, uint32_t ring, uint32_t pbuf,
                                          TcHeader* hdr, uint32_t tmem, TcIter it, int64_t hi) {
  using L = TcSmem<D>;
  const int lane = threadIdx.x & 31;
  const uint32_t S = p.stages, wl = p.wait_limit;
  constexpr uint32_t kIdPV = idesc_e4m3(D, 2 * kMaxG, true, true);
  const uint64_t vd0 = smem_desc(ring + L::kKV, 1024, 1024, 2);
  const uint64_t pd0 = smem_desc(pbuf, 128, 128, 0);
  for (uint32_t j = 0; it.nt > 0; ++j) {
    const uint32_t st = j % S;
    bool ok = tc_wait(smem_addr(&hdr->p_full[j & 1]), (j >> 1) & 1, wl);
    if (ok && j >= 2) ok = tc_wait(smem_addr(&hdr->o_empty[j & 1]), ((j >> 1) - 1) & 1, wl);
    if (!__all_sync(0xffffffffu, ok)) break;
    tc_fence_after_sync();
    if (lane == 0) {
      const uint64_t vd = vd0 + (st * L::kStage >> 4);
      const uint64_t pd = pd0 + ((j & 1) * L::kP >> 4);
      const uint32_t to = tmem + kTcOCol + (j & 1) * 16;
      const int ks = (tc_valid(it) + 31) >> 5;  // rows past the last valid are zero
      umma_e4m3(to, vd, pd, kIdPV, false);
      for (int k = 1; k < ks; ++k)
        umma_e4m3(to, vd + k * (32 * D >> 4), pd + k * (32 * 2 * kMaxG >> 4), kIdPV, true);
      umma_commit(smem_addr(&hdr->o_full[j & 1]));
      umma_commit(smem_addr(&hdr->empty[st]));
    }
    __syncwarp();
    tc_next(p, it, hi);
  }
  if (lane == 0) {
    umma_commit(smem_addr(&hdr->mma_done[1]));
    tc_wait(smem_addr(&hdr->mma_done[1]), 0, wl);
  }
  __syncwarp();
}

// ------------------------------------------------------------- softmax ---
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// The end of a piece for softmax group g (heads 4g .. 4g + 3): sums over
// the chunk's 128 threads, then the normalised output (whole segment) or the
// partial (o, m, l) for the merge kernel, as the other decode kernels write
// them.  Thread t holds d = t.
template <int D>
__device__ __forceinline__ void tc_finish(const DecodeParams& p, TcHeader* hdr, const TcIter& c,
                                          int g, const float (&mf)[kTcGroupHeads],
                                          const float (&lf)[kTcGroupHeads],
                                          const float (&acc)[kTcGroupHeads], uint32_t nfin,
                                          int64_t U, int32_t P) {
  const int lane = threadIdx.x & 31, qd = (threadIdx.x >> 5) & 3;
  const int t = 32 * qd + lane;
  float (*red)[kTcGroupHeads] = hdr->red_l[nfin & 1][g];
  float Lh[kTcGroupHeads];
#pragma unroll
  for (int i = 0; i < kTcGroupHeads; ++i) Lh[i] = warp_sum(lf[i]);
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < kTcGroupHeads; ++i) red[qd][i] = Lh[i];
  tc_group_sync(g);
#pragma unroll
  for (int i = 0; i < kTcGroupHeads; ++i) Lh[i] = (red[0][i] + red[1][i]) + (red[2][i] + red[3][i]);
  const int G = p.group;
  const int h0 = kTcGroupHeads * g;
  if (c.whole) {
    __nv_bfloat16* ob =
        p.out + (static_cast<int64_t>(c.c.b) * p.num_q_heads + c.c.g * G + h0) * D + t;
#pragma unroll
    for (int i = 0; i < kTcGroupHeads; ++i)
      if (h0 + i < G) ob[i * D] = __float2bfloat16_rn(acc[i] / Lh[i]);
    return;
  }
  const int64_t piece = static_cast<int64_t>(blockIdx.x) + c.c.b * p.num_kv_heads + c.c.g;
  float* wo = p.ws_o + (piece * kMaxG + h0) * D + t;
#pragma unroll
  for (int i = 0; i < kTcGroupHeads; ++i) {
    if (h0 + i < G) wo[i * D] = acc[i];
    if (h0 + i < G && t == i) p.ws_ml[piece * kMaxG + h0 + i] = make_float2(mf[i], Lh[i]);
  }
  // the CTA that ends a split segment hands its merge to the merge kernel
  if (g == 0 && t == 0 && c.seg_end == c.c.T)
    p.ws_job[blockIdx.x] = make_int2(c.c.b * p.num_kv_heads + c.c.g,
                                     first_cta(p, U, P, c.useg, c.c.b, c.c.g));
}

// Softmax warps 2-9: group g = (warp - 2) / 4 takes heads 4g .. 4g + 3,
// i.e. columns 8g .. 8g + 7 of S and O.  Thread t = 32 (warp % 4) + lane is
// token t of each chunk (its tensor-memory lane) and d = t of the output.
template <int D>
__device__ __forceinline__ void tc_softmax(const DecodeParams& p, uint32_t ring, uint32_t pbuf,
                                           TcHeader* hdr, uint32_t tmem, TcIter it, int64_t hi,
                                           int64_t U, int32_t P, int g) {
  using L = TcSmem<D>;
  constexpr int H = kTcGroupHeads;
  const int lane = threadIdx.x & 31, qd = (threadIdx.x >> 5) & 3;
  const int t = 32 * qd + lane;
  const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16) + 8 * g;
  const int bshift = p.block_size < kTile ? 3 : 4;  // token -> box
  const uint32_t S = p.stages, wl = p.wait_limit;
  float hm[H], m[H], mt[H], l[H], lold[H];
  float acc[H], macc[H], mc1[H];
#pragma unroll
  for (int i = 0; i < H; ++i) {
    hm[i] = 0.f;
    m[i] = mt[i] = macc[i] = mc1[i] = -INFINITY;
    l[i] = lold[i] = acc[i] = 0.f;
  }
  bool bad = false;
  if (p.stall) bad = !tc_wait(smem_addr(&hdr->stall), 0, wl);  // test hook
  uint32_t j = 0, sg = 0, nfin = 0, st = 0, ph = 0;
  bool have_prev = false, grew1 = false, last1 = false;
  float f1 = 0.f;  // the previous chunk's O unit
  TcIter prev = it;
  for (;;) {
    const bool have = it.nt > 0;
    bool grew = false;
    float f = 0.f;
    if (have) {
      if (it.first) {
        bad |= !tc_wait(smem_addr(&hdr->qready[sg & 1]), (sg >> 1) & 1, wl);
#pragma unroll
        for (int i = 0; i < H; ++i) {
          hm[i] = hdr->hm[sg & 1][H * g + i];
          lold[i] = l[i];
          m[i] = mt[i] = -INFINITY;
          l[i] = 0.f;
        }
        ++sg;
      }
      bad |= !tc_wait(smem_addr(&hdr->full[st]), ph, wl);
      bad |= !tc_wait(smem_addr(&hdr->s_full[j & 1]), (j >> 1) & 1, wl);
      tc_fence_after_sync();  // the MMA's tensor-memory writes before the load
      // tokens t + 128 h of the chunk, h < kTcHalves: S columns 16 h on
      uint32_t sr[kTcHalves][8];  // hi of the group's 4 heads, then their lo
#pragma unroll
      for (int h = 0; h < kTcHalves; ++h) tmem_ld8(tl + (j & 1) * kTcSCols + 16 * h, sr[h]);
      tmem_wait_ld();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&hdr->s_empty[j & 1]));
      const int32_t nvalid = tc_valid(it);
      bool valid[kTcHalves];
      float vs[kTcHalves], x[kTcHalves][H];
      float vsm = 0.f;
      bool gr = false;
#pragma unroll
      for (int h = 0; h < kTcHalves; ++h) {
        const int tok = t + kTcM * h;
        valid[h] = tok < nvalid;
        const int box = tok >> bshift;
        const float ks = hdr->sk[st][box];
        vs[h] = valid[h] ? hdr->sv[st][box] : 0.f;
        vsm = fmaxf(vsm, vs[h]);
        // heads in pairs: s = hi + lo / 16, x = s * k_scale * scale / 2^s
#pragma unroll
        for (int i = 0; i < H; i += 2) {
          const float2 sv = fma2(
              make_float2(__uint_as_float(sr[h][H + i]), __uint_as_float(sr[h][H + i + 1])),
              make_float2(0.0625f, 0.0625f),
              make_float2(__uint_as_float(sr[h][i]), __uint_as_float(sr[h][i + 1])));
          const float2 xv = mul2(sv, mul2(make_float2(ks, ks), make_float2(hm[i], hm[i + 1])));
          x[h][i] = valid[h] ? xv.x : -INFINITY;
          x[h][i + 1] = valid[h] ? xv.y : -INFINITY;
          gr |= x[h][i] > mt[i] || x[h][i + 1] > mt[i + 1];
        }
      }
      const uint32_t wv = __reduce_max_sync(0xffffffffu, __float_as_uint(vsm));  // vs >= 0
      if (lane == 0) hdr->red_v[j & 1][g][qd] = __uint_as_float(wv);
      if (tc_group_popc(g, gr || bad) != 0) {
        if (tc_group_popc(g, bad) != 0) break;  // the group's four warps leave
        // a score passed the running max by more than the slack: the
        // chunk's maxima over its tokens become the new running max
        float mx[H];
#pragma unroll
        for (int i = 0; i < H; ++i) {
          float v = x[0][i];
#pragma unroll
          for (int h = 1; h < kTcHalves; ++h) v = fmaxf(v, x[h][i]);
          mx[i] = warp_max(v);
        }
        if (lane == 0)
#pragma unroll
          for (int i = 0; i < H; ++i) hdr->red_m[g][qd][i] = mx[i];
        tc_group_sync(g);
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const float mn = fmaxf(fmaxf(m[i], fmaxf(hdr->red_m[g][0][i], hdr->red_m[g][1][i])),
                                 fmaxf(hdr->red_m[g][2][i], hdr->red_m[g][3][i]));
          l[i] *= fast_exp2(m[i] - mn);
          m[i] = mn;
          mt[i] = mn + kTcSlack;
        }
        grew = true;
      }
      const float4 rv = *reinterpret_cast<const float4*>(hdr->red_v[j & 1][g]);
      const float vmax = fmaxf(fmaxf(rv.x, rv.y), fmaxf(rv.z, rv.w));
      f = vmax * (1.f / kTcPScale);
      const float rinv = __fdividef(kTcPScale, vmax);
#pragma unroll
      for (int h = 0; h < kTcHalves; ++h) {
        const int tok = t + kTcM * h;
        const float r = vs[h] * rinv;
        float pq[H];
#pragma unroll
        for (int i = 0; i < H; i += 2) {
          const float2 d = add2(make_float2(x[h][i], x[h][i + 1]), make_float2(-m[i], -m[i + 1]));
          const float2 pp = make_float2(fast_exp2(d.x), fast_exp2(d.y));
          const float2 ls = add2(make_float2(l[i], l[i + 1]), pp);
          l[i] = ls.x;
          l[i + 1] = ls.y;
          const float2 q2 = mul2(pp, make_float2(r, r));
          pq[i] = q2.x;
          pq[i + 1] = q2.y;
        }
        uint32_t h0, l0, h1, l1;
        split_e4m3x2(pq[0], pq[1], h0, l0);
        split_e4m3x2(pq[2], pq[3], h1, l1);
        asm volatile("st.shared.v2.b32 [%0], {%1,%2};" ::"r"(pbuf + (j & 1) * L::kP + tok * 16 +
                                                               8 * g),
                     "r"(h0 | (h1 << 16)), "r"(l0 | (l1 << 16))
                     : "memory");
        // V rows past the sequence inside the last 32-token MMA step hold
        // stale bytes (possibly NaN codes): zero them, as P is zero there
        // (with two groups, group 0 the first half of the row, group 1 the
        // second)
        if (!valid[h] && tok < ((nvalid + 31) & ~31)) {
          const bool both = p.group > kTcGroupHeads;
          const uint32_t vrow =
              ring + st * L::kStage + L::kKV + tok * D + (both ? g * (D / 2) : 0);
          for (int o = 0; o < (both ? D / 2 : D); o += 16)
            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(vrow + o), "r"(0)
                         : "memory");
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&hdr->p_full[j & 1]));
    }
    if (have_prev) {
      const uint32_t c = j - 1;
      bad |= !tc_wait(smem_addr(&hdr->o_full[c & 1]), (c >> 1) & 1, wl);
      tc_fence_after_sync();
      uint32_t orr[8];
      tmem_ld8(tl + kTcOCol + (c & 1) * 16, orr);
      tmem_wait_ld();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&hdr->o_empty[c & 1]));
      if (grew1)
#pragma unroll
        for (int i = 0; i < H; ++i) {
          acc[i] *= fast_exp2(macc[i] - mc1[i]);
          macc[i] = mc1[i];
        }
#pragma unroll
      for (int i = 0; i < H; ++i)
        acc[i] = fmaf(f1, fmaf(__uint_as_float(orr[H + i]), 0.0625f, __uint_as_float(orr[i])),
                      acc[i]);
      if (last1) {
        // the chunk opened by this iteration (if any) began a new piece
        const bool moved = have && it.first;
        float lf[H];
#pragma unroll
        for (int i = 0; i < H; ++i) lf[i] = moved ? lold[i] : l[i];
        tc_finish<D>(p, hdr, prev, g, mc1, lf, acc, nfin++, U, P);
#pragma unroll
        for (int i = 0; i < H; ++i) {
          acc[i] = 0.f;
          macc[i] = -INFINITY;
        }
      }
    }
    if (!have) break;
#pragma unroll
    for (int i = 0; i < H; ++i) mc1[i] = m[i];
    grew1 = grew;
    f1 = f;
    last1 = tc_last(it);
    prev = it;
    have_prev = true;
    tc_next(p, it, hi);
    ++j;
    if (++st == S) {
      st = 0;
      ph ^= 1;
    }
  }
}

// --------------------------------------------------------------- kernel ---
template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_decode_tc_fp8_kernel(const __grid_constant__ CUtensorMap tm_q,
                               const __grid_constant__ CUtensorMap tm_k,
                               const __grid_constant__ CUtensorMap tm_v,
                               const DecodeParams p) {
  using L = TcSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_addr(smem_raw);
  if ((base & 1023u) || p.stages < 2 || p.stages > kTcMaxStages || p.skip != 0 ||
      p.pf_o != nullptr || p.k_new != nullptr) {
    if (threadIdx.x == 0) flag_error(PA_DEVERR_LAUNCH);
    return;
  }
  const uint32_t ring = base;
  const uint32_t qbuf = ring + p.stages * L::kStage;
  const uint32_t q8buf = qbuf + 2 * L::kQ;
  const uint32_t pbuf = q8buf + 2 * L::kQ8;
  TcHeader* hdr = reinterpret_cast<TcHeader*>(smem_raw + (pbuf - base) + 2 * L::kP);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_addr(&hdr->full[s]), kTcCopyWarps);
      mbar_init(smem_addr(&hdr->empty[s]), 1);
    }
    // softmax warps that take part: group 1 only when the GQA group has
    // more than 4 heads (its heads would all be past the group)
    const uint32_t nsoft = p.group > kTcGroupHeads ? kTcSoftWarps : kTcSoftWarps / 2;
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&hdr->qfull[s]), 1);
      mbar_init(smem_addr(&hdr->qempty[s]), 1);
      mbar_init(smem_addr(&hdr->qready[s]), 1);
      mbar_init(smem_addr(&hdr->s_full[s]), 1);
      mbar_init(smem_addr(&hdr->s_empty[s]), nsoft);
      mbar_init(smem_addr(&hdr->p_full[s]), nsoft);
      mbar_init(smem_addr(&hdr->o_full[s]), 1);
      mbar_init(smem_addr(&hdr->o_empty[s]), nsoft);
    }
    mbar_init(smem_addr(&hdr->mma_done[0]), 1);
    mbar_init(smem_addr(&hdr->mma_done[1]), 1);
    mbar_init(smem_addr(&hdr->stall), 1);
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&hdr->tmem), kTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = hdr->tmem;
  // The work split reads only seq_lens, before the wait for the previous
  // grid (as in the other decode kernels); every warp computes it.
  int64_t U, lo, hi;
  int32_t P;
  Cursor c;
  const bool mine = my_range(p, U, P, lo, hi, c);
  pdl_wait();
  pdl_trigger();
  if (p.ws_job != nullptr && threadIdx.x == 32) p.ws_job[blockIdx.x] = make_int2(-1, -1);
  if (mine) {
    TcIter it;
    it.c = c;
    it.u = lo;
    tc_open_piece(it, hi);
    // warps: 0 and 11.. copies, 1 QK MMAs, 2-9 softmax, 10 PV MMAs
    if (warp == 0 || warp > 10) {
      const int part = warp == 0 ? 0 : warp - 10;
      tc_produce<D>(p, &tm_q, (part & 1) ? &tm_v : &tm_k, part, ring, qbuf, hdr, it, hi);
    } else if (warp == 1) {
      tc_mma_qk<D>(p, ring, qbuf, q8buf, hdr, tmem, it, hi);
    } else if (warp == 10) {
      tc_mma_pv<D>(p, ring, pbuf, hdr, tmem, it, hi);
    } else if (((warp - 2) >> 2) * kTcGroupHeads < p.group) {
      tc_softmax<D>(p, ring, pbuf, hdr, tmem, it, hi, U, P, (warp - 2) >> 2);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, kTcTmemCols);
}

}  // namespace pa
