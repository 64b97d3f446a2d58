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
//   (b, g, tile), and each persistent CTA of P owns a contiguous run of it.
//   The runs balance cost, not tiles: a segment costs its tiles plus a
//   fixed charge for its query copy, first table batch and finish, so a
//   CTA that meets many short segments takes fewer tiles.  Long contexts
//   split into at most P pieces in total (split-K).  A piece that covers
//   a whole segment writes the output directly; otherwise it writes an
//   unnormalised partial (o, m, l) that the merge kernel combines by
//   log-sum-exp.  Split points depend only on seq_lens, so the output does
//   not depend on which physical blocks the tables name.
// * Copies: 2D TMA boxes of each tile's K and V rows (128 bytes wide, 128B
//   swizzle; 64B for FP8 d=64) into a ring of shared-memory stages, one
//   mbarrier per stage, plus the G query rows of each new segment.  Block-
//   table entries arrive 32 blocks at a time from one coalesced warp load,
//   the next batch (and its FP8 scales) loaded ahead.
// * CTA shape per instantiation.  bf16: 2 warps, a copy warp and a math
//   warp, 8 CTAs per SM -- under full HBM load a TMA issue stalls its
//   thread for hundreds of cycles, and the copy warp absorbs that.  FP8:
//   the math per byte is ~2.5x heavier, so every warp computes: 1-warp
//   CTAs (16 per SM) that top their ring up after each tile.
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
  int2* ws_job;   // [P]: (segment, first CTA) of the split segment that
                  // CTA finishes, else (-1, -1)
  // Fused append (bf16 caches; null when off): sequence b's new token
  // k_new/v_new[b][Hkv][D] goes to slot_mapping[b] (< 0: none), which must
  // be the slot the table gives position seq_lens[b] - 1.
  const uint8_t* k_new;
  const uint8_t* v_new;
  const int64_t* slot_mapping;
  uint8_t* k_cache;
  uint8_t* v_cache;
  // Cascade (null / 0 when off): this call's tiles start at token `skip` of
  // every sequence, and the attention over tokens [0, skip) arrives as a
  // partial per (sequence, query head) to fold in: pf_o[B][Hq][D]
  // unnormalised, pf_ml[B][Hq] (max in log2 units, sum).
  int32_t skip;
  const float* pf_o;
  const float2* pf_ml;
  int32_t num_seqs, num_q_heads, num_kv_heads, group, block_size, log2_bs;
  int32_t max_blocks, num_blocks;
  int32_t rows_total;  // num_blocks * num_kv_heads * block_size
  float scale_log2;    // softmax scale * log2(e)
  int32_t num_ctas;    // P
  int32_t seg_cost;    // work split: units charged per segment (a work unit is kUnit)
  int32_t tile_log2;   // work unit of the split: 2^tile_log2 16-token tiles (0 but in
                       // kernels that take a segment in larger chunks)
  int32_t stages;      // ring depth
  // Bounded waits: polls before a math-warp wait gives up (PA_DEVERR_TIMEOUT;
  // the copy warp's waits keep the fixed default bound: a run-time bound
  // there slowed the block-size-8 decode by 47%, measured).  stall != 0 (a
  // test hook) makes the math warp first wait on a barrier nothing arrives
  // at, so the timeout path runs deterministically.
  uint32_t wait_limit;
  int32_t stall;
};

// ------------------------------------------------ shared memory layout ---
// [query slots | stage ring | header].  A bf16 tile is D/64 slabs of 16
// rows x 128 bytes, an FP8 tile 16 rows x D bytes, both as the TMA's 128B
// (64B for FP8 d=64) swizzle writes them: the 8 rows of an ldmatrix hit 8
// different bank groups.  Query slots and stages are multiples of 1024
// bytes, so every box starts 1024-aligned.
constexpr int kQSlots = 2;
constexpr int kMaxStages = 24;

template <int D, bool FP8>
struct Smem {
  static constexpr int kSlabBytes = FP8 ? kTile * D : kTile * 128;  // one box
  static constexpr int kSlabs = FP8 ? 1 : D / 64;
  static constexpr int kKVBytes = kSlabs * kSlabBytes;  // K (or V) of a tile
  static constexpr int kStageBytes = 2 * kKVBytes;
  static constexpr int kQSlabBytes = 8 * 128;           // 8 rows x 64 bf16
  static constexpr int kQBytes = (D / 64) * kQSlabBytes;
  static_assert(kStageBytes % 1024 == 0 && kQBytes % 1024 == 0, "alignment");
};

struct Header {
  uint64_t full[kMaxStages];   // stage landed
  uint64_t empty[kMaxStages];  // stage read (two-warp CTAs)
  uint64_t qfull[kQSlots];     // query slot landed
  uint64_t qempty[kQSlots];    // query slot read (two-warp CTAs)
  uint64_t stall;              // never arrived at (the stall test hook waits on it)
  float4 scales[kMaxStages];  // FP8: (k_scale row g, k_scale row g+8, v_scale ...)
};

template <int D, bool FP8>
__host__ __device__ constexpr size_t decode_smem_bytes(int stages) {
  return static_cast<size_t>(kQSlots) * Smem<D, FP8>::kQBytes +
         static_cast<size_t>(stages) * Smem<D, FP8>::kStageBytes + sizeof(Header);
}

__device__ __forceinline__ int32_t cdiv16(int32_t n) { return (n + 15) >> 4; }

// Tiles of a sequence of n tokens in this call (its tokens from `skip` on).
__device__ __forceinline__ int32_t seg_tiles(const DecodeParams& p, int32_t n) {
  return n > p.skip ? (cdiv16(n - p.skip) + (1 << p.tile_log2) - 1) >> p.tile_log2 : 0;
}

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

// Move to the first tile of the next non-empty segment.
__device__ __forceinline__ void next_segment(const DecodeParams& p, Cursor& c) {
  c.tile = 0;
  if (++c.g < p.num_kv_heads) return;
  c.g = 0;
  do {
    ++c.b;
    c.n = c.b < p.num_seqs ? clamp_len(p, p.seq_lens[c.b]) : 1;
    c.T = seg_tiles(p, c.n);
  } while (c.T == 0);
}

// The cost-weighted split.  A tile costs kUnit units and every segment
// (b, g) seg_cost more, charged just before its first tile: the query
// copy, the first table batch and the finish are paid once per segment.
// So tile t of segment s = b*Hkv + g has its first unit at
//   kUnit * (flat index of the tile) + seg_cost * (s + 1),
// and the list holds U = kUnit * W + seg_cost * B * Hkv units.  CTA c of P
// takes the units [U*c/P, U*(c+1)/P) and with them the tiles whose first
// unit lies there, a contiguous run [lo, hi) of the flat list.  With
// P <= W every range spans at least kUnit units, so a CTA strictly inside
// a split segment always holds some of its tiles; a range that falls in
// the units charged between two segments holds none.
constexpr int kUnit = 8;

// a / b for non-negative a, b > 0, in 32 bits when both fit.
__device__ __forceinline__ int64_t div_nn(int64_t a, int64_t b) {
  if (((a | b) >> 31) == 0)
    return static_cast<uint32_t>(a) / static_cast<uint32_t>(b);
  return a / b;
}

// a * c / P for a >= 0 and 0 <= c <= P (no 64-bit division when a fits in
// 31 bits and P is small): a = qP + r, so a*c/P = q*c + r*c/P.
__device__ __forceinline__ int64_t mul_div(int64_t a, int32_t c, int32_t P) {
  if ((a >> 31) == 0 && P <= 46340) {
    const uint32_t u = static_cast<uint32_t>(a), pp = static_cast<uint32_t>(P),
                   cc = static_cast<uint32_t>(c);
    return static_cast<int64_t>(u / pp) * cc + (u % pp) * cc / pp;
  }
  return a * c / P;
}

// Warp-collective: 128 sequences from b00, lane l holding b00 + 4l + k.
struct Chunk {
  int32_t n[4];  // clamped lengths (0 past the batch)
  int64_t excl;  // tiles (all heads) of the chunk's sequences before this lane's
  int64_t sum;   // tiles of this lane's four
  int64_t total; // tiles of the chunk
};

__device__ __forceinline__ void load_chunk(const DecodeParams& p, int32_t b00, Chunk& ch) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int32_t b = b00 + 4 * lane + k;
    ch.n[k] = b < p.num_seqs ? clamp_len(p, p.seq_lens[b]) : 0;
  }
  int64_t s = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) s += seg_tiles(p, ch.n[k]);
  s *= p.num_kv_heads;
  int64_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if ((threadIdx.x & 31) >= o) incl += y;
  }
  ch.sum = s;
  ch.excl = incl - s;
  ch.total = __shfl_sync(0xffffffffu, incl, 31);
}

// Warp-collective: if unit x lies in chunk ch (base = tiles before it),
// the number of tiles whose first unit is below x, and, if want, the
// segment cursor there (before any move past a segment's end).
__device__ __forceinline__ bool find_in_chunk(const DecodeParams& p, const Chunk& ch,
                                              int32_t b00, int64_t base, int64_t x,
                                              int64_t& t, Cursor* c) {
  const int lane = threadIdx.x & 31;
  const int64_t A = p.seg_cost;
  const int32_t H = p.num_kv_heads;
  const int32_t b0 = b00 + 4 * lane;
  const int32_t nthrough = min(b0 + 4, p.num_seqs);  // sequences through this lane's
  const int64_t uthrough = kUnit * (base + ch.excl + ch.sum) + A * H * nthrough;
  const unsigned m = __ballot_sync(0xffffffffu, b0 < p.num_seqs && uthrough > x);
  if (m == 0u) return false;
  const int L = __ffs(m) - 1;
  int64_t before = base + __shfl_sync(0xffffffffu, ch.excl, L);
  int32_t n[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) n[k] = __shfl_sync(0xffffffffu, ch.n[k], L);
  int32_t b = b00 + 4 * L;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int32_t T = seg_tiles(p, n[k]);
    const int64_t seg = kUnit * static_cast<int64_t>(T) + A;  // units of one head
    const int64_t rem = x - (kUnit * before + A * H * b);
    if (k == 3 || rem < seg * H) {
      const int64_t g = div_nn(rem, seg);
      const int64_t r = rem - g * seg;
      const int64_t j = r <= A ? 0 : (r - A + kUnit - 1) / kUnit;
      t = before + g * T + j;
      if (c != nullptr) {
        c->b = b;
        c->n = n[k];
        c->T = T;
        c->g = T == 0 ? H - 1 : static_cast<int32_t>(g);  // an empty sequence: past its last head
        c->tile = T == 0 ? 0 : static_cast<int32_t>(j);
      }
      return true;
    }
    before += static_cast<int64_t>(H) * T;
    ++b;
  }
  return true;  // not reached
}

// This CTA's range [lo, hi) of the flat tile list and the cursor at lo
// (U units over P participating CTAs); false if it holds no tile.  With
// fewer tiles than CTAs only the first W CTAs take part.  Reads only
// seq_lens: once for up to 128 sequences.
__device__ __forceinline__ bool my_range(const DecodeParams& p, int64_t& U, int32_t& P,
                                         int64_t& lo, int64_t& hi, Cursor& c) {
  Chunk ch;
  load_chunk(p, 0, ch);
  int64_t W = ch.total;
  for (int32_t b00 = 128; b00 < p.num_seqs; b00 += 128) {
    Chunk more;
    load_chunk(p, b00, more);
    W += more.total;
  }
  if (W == 0) return false;
  U = kUnit * W + static_cast<int64_t>(p.seg_cost) * p.num_kv_heads * p.num_seqs;
  P = static_cast<int32_t>(min(static_cast<int64_t>(p.num_ctas), W));
  const int32_t cta = static_cast<int32_t>(blockIdx.x);
  if (cta >= P) return false;
  const int64_t x0 = mul_div(U, cta, P), x1 = mul_div(U, cta + 1, P);
  bool f0 = false, f1 = false;
  lo = hi = W;  // a bound past every sequence's units
  int64_t base = 0;
  for (int32_t b00 = 0; b00 < p.num_seqs && !(f0 && f1); b00 += 128) {
    if (b00 > 0) load_chunk(p, b00, ch);
    if (!f0) f0 = find_in_chunk(p, ch, b00, base, x0, lo, &c);
    if (!f1) f1 = find_in_chunk(p, ch, b00, base, x1, hi, nullptr);
    base += ch.total;
  }
  if (lo >= hi) return false;
  // a bound at a segment's end (or in an empty sequence) opens the next one
  if (c.T == 0 || c.tile == c.T) next_segment(p, c);
  return true;
}

// Index of the CTA holding the first tile of segment (b, g), flat tile f.
__device__ __forceinline__ int32_t first_cta(const DecodeParams& p, int64_t U, int32_t P,
                                             int64_t f, int32_t b, int32_t g) {
  const int64_t F = kUnit * f + static_cast<int64_t>(p.seg_cost) *
                                    (static_cast<int64_t>(b) * p.num_kv_heads + g + 1);
  return static_cast<int32_t>(((F + 1) * P - 1) / U);
}

// ---------------------------------------------------------- issue side ---
struct Maps {
  const CUtensorMap* q;
  const CUtensorMap* k;
  const CUtensorMap* v;
};

struct Bufs {
  uint32_t q, ring;  // shared addresses of the query slots and the ring
  Header* hdr;
};

// Table batch: lane l holds the entry of block (l & (rpt - 1)) of tile
// tb + l / rpt, rpt = blocks per tile (2 for block_size 8, else 1).
struct Loader {
  Cursor c;          // next tile to issue
  int64_t u;         // its flat index
  int32_t seg_end;   // end of this CTA's part of c's segment
  int32_t tb;        // first tile of the table batch held (-1: none)
  int32_t e;         // this lane's table entry
  int32_t ne;        // the same for the next batch, loaded ahead
  float ks, vs;      // FP8: scales of e for head g
  float nks, nvs;    // FP8: scales of ne, loaded mid-batch
  uint32_t it;       // tiles issued
  uint32_t qn;       // query slots filled (segments begun)
  bool fresh;        // the next tile opens a segment
  int64_t slot;      // fused append: slot of the segment's new token
  uint4 row;         // fused append: this lane's 16 bytes of its K|V row
};

// log2 of the blocks per 16-token tile
__device__ __forceinline__ int rpt_log2(const DecodeParams& p) {
  return p.block_size < kTile ? 1 : 0;
}

// This lane's table entry in the batch that starts at tile t (-1 past the
// end of the CTA's part of the segment or of the sequence).
__device__ __forceinline__ int32_t fetch_entry(const DecodeParams& p, const Loader& ld,
                                               int32_t t) {
  const int lane = threadIdx.x & 31;
  const int lr = rpt_log2(p);
  const int32_t tile = t + (lane >> lr);
  const int32_t tok = p.skip + tile * kTile + (lane & ((1 << lr) - 1)) * p.block_size;
  if (tile >= ld.seg_end || tok >= ld.c.n) return -1;
  return p.block_tables[static_cast<int64_t>(ld.c.b) * p.max_blocks + (tok >> p.log2_bs)];
}

// FP8 scales of block x for head g (1 for ids out of range).
__device__ __forceinline__ void fetch_scales(const DecodeParams& p, int32_t g, int32_t x,
                                             float& k, float& v) {
  k = v = 1.f;
  if (x >= 0 && x < p.num_blocks) {
    k = p.k_scale[static_cast<int64_t>(x) * p.num_kv_heads + g];
    v = p.v_scale[static_cast<int64_t>(x) * p.num_kv_heads + g];
  }
}

// Warp-collective: make the table entries (and FP8 scales) of tile
// ld.c.tile available.  The next batch's entries are loaded one batch
// ahead and their scales half a batch ahead, so only the first batch of a
// segment waits on memory.
template <bool FP8>
__device__ __forceinline__ void advance_table(const DecodeParams& p, Loader& ld) {
  const int32_t t = ld.c.tile;
  const int32_t per = 32 >> rpt_log2(p);  // tiles per batch
  if (ld.tb < 0) {
    ld.e = fetch_entry(p, ld, t);
    if (FP8) fetch_scales(p, ld.c.g, ld.e, ld.ks, ld.vs);
    ld.ne = fetch_entry(p, ld, t + per);
    ld.tb = t;
  } else if (t - ld.tb == per) {
    ld.e = ld.ne;
    if (FP8) {
      ld.ks = ld.nks;
      ld.vs = ld.nvs;
    }
    ld.ne = fetch_entry(p, ld, t + per);
    ld.tb = t;
  }
  if (FP8 && t - ld.tb == per / 2) fetch_scales(p, ld.c.g, ld.ne, ld.nks, ld.nvs);
}

// Lane 0: the query rows of segment c into slot `slot` (8 rows from
// b*Hq + g*G; rows past the group are ignored, rows past the tensor read
// zeros).
template <int D, bool FP8>
__device__ __forceinline__ void copy_query(const DecodeParams& p, const Maps& tm,
                                           const Bufs& sb, const Cursor& c, uint32_t slot) {
  using L = Smem<D, FP8>;
  const uint32_t bar = smem_addr(&sb.hdr->qfull[slot]);
  mbar_arrive_expect_tx(bar, L::kQBytes);
  const int32_t row = c.b * p.num_q_heads + c.g * p.group;
#pragma unroll
  for (int sl = 0; sl < D / 64; ++sl)
    tma_load_2d(sb.q + slot * L::kQBytes + sl * L::kQSlabBytes, tm.q, sl * 64, row, bar);
}

// Lane 0: K and V rows of tile c.tile into `stage`, one box per block (two
// for block_size 8).  An invalid block id reads rows past the tensor, which
// the TMA fills with zeros.
template <int D, bool FP8>
__device__ __forceinline__ void copy_tile(const DecodeParams& p, const Maps& tm,
                                          const Bufs& sb, const Cursor& c, uint32_t stage,
                                          int32_t b0, int32_t b1) {
  using L = Smem<D, FP8>;
  const int32_t tok = p.skip + c.tile * kTile;
  const int box_rows = p.block_size < kTile ? p.block_size : kTile;
  const uint32_t box_bytes = static_cast<uint32_t>(box_rows) * (FP8 ? D : 128);
  const int nbox = (p.block_size < kTile && tok + p.block_size < c.n) ? 2 : 1;
  const uint32_t bar = smem_addr(&sb.hdr->full[stage]);
  mbar_arrive_expect_tx(bar, 2u * nbox * L::kSlabs * box_bytes);
  const uint32_t kdst = sb.ring + stage * L::kStageBytes;
  const uint32_t vdst = kdst + L::kKVBytes;
  for (int bx = 0; bx < nbox; ++bx) {
    const int32_t blk = bx == 0 ? b0 : b1;
    int32_t row;  // row = (blk * Hkv + g) * bs + offset
    if (blk < 0 || blk >= p.num_blocks) {
      flag_error(PA_DEVERR_BAD_BLOCK_ID);
      row = p.rows_total;  // out of the tensor: zero fill
    } else {
      const int32_t off = p.block_size >= kTile ? (tok & (p.block_size - 1)) : 0;
      row = (blk * p.num_kv_heads + c.g) * p.block_size + off;
    }
    const uint32_t sub = static_cast<uint32_t>(bx) * box_bytes;
#pragma unroll
    for (int sl = 0; sl < L::kSlabs; ++sl) {
      tma_load_2d(kdst + sl * L::kSlabBytes + sub, tm.k, sl * 64, row, bar);
      tma_load_2d(vdst + sl * L::kSlabBytes + sub, tm.v, sl * 64, row, bar);
    }
  }
}

// Fused append, at the start of segment (b, g): load the slot of sequence
// b's new token and, lane l < 2 * D / 8, 16 bytes of its K (l < D / 8) or
// V row for head g.  Used only at the segment's last tile.
template <int D>
__device__ __forceinline__ void fetch_new_token(const DecodeParams& p, Loader& ld) {
  constexpr int kChunks = D * 2 / 16;
  const int lane = threadIdx.x & 31;
  ld.slot = p.slot_mapping[ld.c.b];
  if (lane < 2 * kChunks) {
    const int kv = lane / kChunks, ch = lane % kChunks;
    const int64_t src = (static_cast<int64_t>(ld.c.b) * p.num_kv_heads + ld.c.g) * (D * 2) + ch * 16;
    ld.row = *reinterpret_cast<const uint4*>((kv ? p.v_new : p.k_new) + src);
  }
}

// Warp-collective, before the copy of the segment's last tile: store the
// new token's K and V rows of head g at its slot, then fence so the tile's
// TMA read sees them.  Only this CTA reads that tile, and copy-on-write
// keeps every appended slot private to its sequence.  A slot that is not
// where the table puts position n - 1 flags PA_DEVERR_BAD_SLOT and is not
// written.
template <int D>
__device__ __forceinline__ void store_new_token(const DecodeParams& p, const Loader& ld,
                                                int32_t b0, int32_t b1) {
  constexpr int kChunks = D * 2 / 16;
  const int lane = threadIdx.x & 31;
  if (ld.slot < 0) return;
  const int32_t pos = ld.c.n - 1;
  const int32_t blk = (p.block_size < kTile && (pos & (kTile - 1)) >= p.block_size) ? b1 : b0;
  const int32_t off = pos & (p.block_size - 1);
  if (blk < 0 || blk >= p.num_blocks ||
      ld.slot != static_cast<int64_t>(blk) * p.block_size + off) {
    if (lane == 0) flag_error(PA_DEVERR_BAD_SLOT);
    return;
  }
  if (lane < 2 * kChunks) {
    const int kv = lane / kChunks, ch = lane % kChunks;
    const int64_t dst =
        ((static_cast<int64_t>(blk) * p.num_kv_heads + ld.c.g) * p.block_size + off) * (D * 2) +
        ch * 16;
    *reinterpret_cast<uint4*>((kv ? p.v_cache : p.k_cache) + dst) = ld.row;
    fence_proxy_async_global();
  }
  __syncwarp();
}

// FP8 version of store_new_token (block_size <= 16, so the tile holds the
// whole block of the new token): lane l < 2 * D / 8 holds 8 bf16 values of
// the K (l < D / 8) or V row.  With the token's own scale s_t = absmax /
// 448: offset 0 sets the block's scale to s_t (1 for a zero row); a larger
// s_t raises it and requantises the block's earlier rows through fp32
// (decode * old / new, RNE satfinite); then the row is e4m3(x / scale).
// Each lane owns the same 8 bytes of every row.  `sc` (this tile's scales:
// x / y = K of the first / second block, z / w = V) gets the new scale.
// The new row is loaded here rather than at the segment's start: the
// single-warp FP8 kernel has no registers to keep it live across the tiles.
template <int D>
__device__ __forceinline__ void store_new_token_fp8(const DecodeParams& p, const Cursor& c,
                                                 int32_t b0, int32_t b1, float4& sc) {
  constexpr int kChunks = D * 2 / 16;  // 16-byte bf16 chunks per row = lanes per K|V
  const int lane = threadIdx.x & 31;
  Loader ld;
  ld.c = c;
  ld.slot = p.slot_mapping[c.b];
  ld.row = make_uint4(0u, 0u, 0u, 0u);
  if (lane < 2 * kChunks) {
    const int kv = lane / kChunks, ch = lane % kChunks;
    const int64_t src = (static_cast<int64_t>(c.b) * p.num_kv_heads + c.g) * (D * 2) + ch * 16;
    ld.row = *reinterpret_cast<const uint4*>((kv ? p.v_new : p.k_new) + src);
  }
  if (ld.slot < 0) return;
  const int32_t pos = ld.c.n - 1;
  const bool second = p.block_size < kTile && (pos & (kTile - 1)) >= p.block_size;
  const int32_t blk = second ? b1 : b0;
  const int32_t off = pos & (p.block_size - 1);
  if (blk < 0 || blk >= p.num_blocks ||
      ld.slot != static_cast<int64_t>(blk) * p.block_size + off) {
    if (lane == 0) flag_error(PA_DEVERR_BAD_SLOT);
    return;
  }
  const bool active = lane < 2 * kChunks;
  const int kv = lane / kChunks, ch = lane % kChunks;
  float x[8];
  float a = 0.f;
  if (active) {
    const uint32_t w4[4] = {ld.row.x, ld.row.y, ld.row.z, ld.row.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack_bf16x2(w4[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
      a = fmaxf(a, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  // absmax over the K lanes and over the V lanes (groups of kChunks lanes)
#pragma unroll
  for (int o = 1; o < kChunks; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const int64_t sidx = static_cast<int64_t>(blk) * p.num_kv_heads + ld.c.g;
  float* scale = const_cast<float*>(kv ? p.v_scale : p.k_scale) + sidx;
  const float old = active ? *scale : 1.f;
  const float st = __fdiv_rn(a, 448.f);
  float nw = old;
  uint8_t* rows = (kv ? p.v_cache : p.k_cache) +
                  (static_cast<int64_t>(blk) * p.num_kv_heads + ld.c.g) * p.block_size * D + ch * 8;
  if (off == 0) {
    nw = a == 0.f ? 1.f : st;
  } else if (st > old) {
    nw = st;
    if (active)
      for (int32_t r = 0; r < off; ++r) {
        uint2* q = reinterpret_cast<uint2*>(rows + static_cast<int64_t>(r) * D);
        uint2 c = *q;
        uint32_t cw[2] = {c.x, c.y};
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          uint32_t out = 0;
#pragma unroll
          for (int bt = 0; bt < 4; ++bt) {
            const __half_raw hr =
                __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(cw[w] >> (8 * bt)),
                                        __NV_E4M3);
            const float y = __fmul_rn(__half2float(__half(hr)), old);
            out |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fdiv_rn(y, nw), __NV_SATFINITE,
                                                               __NV_E4M3))
                   << (8 * bt);
          }
          cw[w] = out;
        }
        *q = make_uint2(cw[0], cw[1]);
      }
  }
  if (active) {
    uint32_t cw[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i)
      cw[i >> 2] |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fdiv_rn(x[i], nw),
                                                                __NV_SATFINITE, __NV_E4M3))
                    << (8 * (i & 3));
    *reinterpret_cast<uint2*>(rows + static_cast<int64_t>(off) * D) = make_uint2(cw[0], cw[1]);
    if (ch == 0) *scale = nw;
    fence_proxy_async_global();
  }
  // this tile's scales for the consumer: K from lane 0, V from lane kChunks
  const float nk = __shfl_sync(0xffffffffu, nw, 0);
  const float nv = __shfl_sync(0xffffffffu, nw, kChunks);
  if (second) {
    sc.y = nk;
    sc.w = nv;
  } else {
    sc.x = nk;
    sc.z = nv;
    if (p.block_size >= kTile || !(b1 >= 0 && b1 < p.num_blocks)) {
      sc.y = nk;  // one block in the tile (or the second is absent)
      sc.w = nv;
    }
  }
  __syncwarp();
}

// Warp-collective: issue the loader's next tile (and, if it opens a
// segment, the segment's query rows) into the next stage, then advance
// the loader.  The caller has made sure the stage and query slot are free.
template <int D, bool FP8, bool kAppend = true>
__device__ __forceinline__ void issue_tile(const DecodeParams& p, const Maps& tm,
                                           const Bufs& sb, Loader& ld, int64_t hi) {
  const int lane = threadIdx.x & 31;
  if (ld.fresh) {
    if (lane == 0) copy_query<D, FP8>(p, tm, sb, ld.c, ld.qn % kQSlots);
    ++ld.qn;
    ld.fresh = false;
    if (!FP8 && p.k_new != nullptr) fetch_new_token<D>(p, ld);
  }
  advance_table<FP8>(p, ld);
  const int lr = rpt_log2(p);
  const int j = (ld.c.tile - ld.tb) << lr;  // lane of the tile's first block
  const int32_t b0 = __shfl_sync(0xffffffffu, ld.e, j);
  const int32_t b1 = __shfl_sync(0xffffffffu, ld.e, (j + lr) & 31);  // bs 8: second block
  const uint32_t stage = ld.it % p.stages;
  if (FP8) {
    float4 sc;
    sc.x = __shfl_sync(0xffffffffu, ld.ks, j);
    sc.y = __shfl_sync(0xffffffffu, ld.ks, (j + lr) & 31);
    sc.z = __shfl_sync(0xffffffffu, ld.vs, j);
    sc.w = __shfl_sync(0xffffffffu, ld.vs, (j + lr) & 31);
    // an absent (or unusable) second block takes the first one's scales,
    // so the V-scale ratios of the tile stay 1
    if (!(b1 >= 0 && b1 < p.num_blocks)) {
      sc.y = sc.x;
      sc.w = sc.z;
    }
    // written before the stage's arrive, read after its completion
    if (kAppend && p.k_new != nullptr && ld.c.tile == ld.c.T - 1)
      store_new_token_fp8<D>(p, ld.c, b0, b1, sc);
    if (lane == 0) sb.hdr->scales[stage] = sc;
  }
  if (!FP8 && p.k_new != nullptr && ld.c.tile == ld.c.T - 1) store_new_token<D>(p, ld, b0, b1);
  if (lane == 0) copy_tile<D, FP8>(p, tm, sb, ld.c, stage, b0, b1);
  ++ld.it;
  ++ld.u;
  if (++ld.c.tile == ld.seg_end && ld.u < hi) {
    next_segment(p, ld.c);
    ld.seg_end = static_cast<int32_t>(min(static_cast<int64_t>(ld.c.T), hi - ld.u));
    ld.tb = -1;
    ld.fresh = true;
  }
}

// The loader at flat tile lo (cursor c) of a CTA owning [lo, hi).
__device__ __forceinline__ void loader_init(int64_t lo, int64_t hi, const Cursor& c,
                                            Loader& ld) {
  ld.c = c;
  ld.u = lo;
  ld.seg_end = static_cast<int32_t>(min(static_cast<int64_t>(ld.c.T), ld.c.tile + (hi - lo)));
  ld.tb = -1;
  ld.e = ld.ne = -1;
  ld.ks = ld.vs = ld.nks = ld.nvs = 1.f;
  ld.it = ld.qn = 0;
  ld.fresh = true;
  ld.slot = -1;
  ld.row = make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ bool can_issue(const DecodeParams& p, const Loader& ld,
                                          int64_t hi, uint32_t used, uint32_t qread) {
  return ld.u < hi && ld.it - used < static_cast<uint32_t>(p.stages) &&
         (!ld.fresh || ld.qn - qread < static_cast<uint32_t>(kQSlots));
}

// Single-warp CTA: issue tiles while a stage is free (`used` = tiles
// consumed) and, for a tile that opens a segment, a query slot is free
// (`qread` = slots read).  The warp has synchronised after its last reads
// of the bytes these copies overwrite; the proxy fence orders those reads
// before the TMA writes.
template <int D, bool FP8, bool kAppend>
__device__ __forceinline__ void top_up(const DecodeParams& p, const Maps& tm, const Bufs& sb,
                                       Loader& ld, int64_t hi, uint32_t used, uint32_t qread) {
  if (!can_issue(p, ld, hi, used, qread)) return;
  if ((threadIdx.x & 31) == 0) fence_proxy_async_smem();
  do {
    issue_tile<D, FP8, kAppend>(p, tm, sb, ld, hi);
  } while (can_issue(p, ld, hi, used, qread));
  __syncwarp();
}

// Two-warp CTA, copy warp: issue every tile of [lo, hi) as soon as the
// math warp has released its stage (and query slot).
template <int D, bool FP8>
__device__ __forceinline__ void produce(const DecodeParams& p, const Maps& tm, const Bufs& sb,
                                        Loader& ld, int64_t hi) {
  const int lane = threadIdx.x & 31;
  const uint32_t S = p.stages;
  bool ok = true;
  while (ld.u < hi) {
    if (lane == 0) {
      if (ld.fresh && ld.qn >= kQSlots)
        ok = mbar_wait(smem_addr(&sb.hdr->qempty[ld.qn % kQSlots]), (ld.qn / kQSlots - 1) & 1);
      if (ok && ld.it >= S)
        ok = mbar_wait(smem_addr(&sb.hdr->empty[ld.it % S]), (ld.it / S - 1) & 1);
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    issue_tile<D, FP8>(p, tm, sb, ld, hi);
  }
  // No copy may target shared memory after the CTA exits.  On the normal
  // path the math warp has already waited for all of them.
  if (lane == 0) {
    for (uint32_t k = ld.it > S ? ld.it - S : 0; k < ld.it; ++k)
      mbar_wait(smem_addr(&sb.hdr->full[k % S]), (k / S) & 1, 1u << 16);
    for (uint32_t k = ld.qn > kQSlots ? ld.qn - kQSlots : 0; k < ld.qn; ++k)
      mbar_wait(smem_addr(&sb.hdr->qfull[k % kQSlots]), (k / kQSlots) & 1, 1u << 16);
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
    uint32_t c[8];
    e4m3x4_to_f16x2x2(u0, c[0], c[1]);
    e4m3x4_to_f16x2x2(u1, c[2], c[3]);
    e4m3x4_to_f16x2x2(u2, c[4], c[5]);
    e4m3x4_to_f16x2x2(u3, c[6], c[7]);
    mma_f16_zero_c(t0, c[0], c[1], c[2], c[3], pb0, pb1);
    mma_f16_zero_c(t1, c[4], c[5], c[6], c[7], pb0, pb1);
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

// d index of accumulator element (i, q) for lane gq.
template <int D, bool FP8>
__device__ __forceinline__ int acc_d(int i, int q, int gq) {
  if (!FP8) return 16 * i + gq + ((q >> 1) << 3);
  // FP8: m-tile i covers chunk i; rows gq / gq + 8 are d = 16i + 2gq (+1).
  return 16 * i + 2 * gq + (q >> 1);
}

// Query fragments (B operand, n = head, k = d) from a query slot, and for
// FP8 the per-head score multipliers hm0 / hm1 (heads 2tq, 2tq + 1).
template <int D, bool FP8>
__device__ __forceinline__ void load_query(const DecodeParams& p, uint32_t qslot,
                                           uint32_t (&qb)[D / 16][2], float& hm0,
                                           float& hm1) {
  using L = Smem<D, FP8>;
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  hm0 = hm1 = p.scale_log2;
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
}

// Write a finished piece of segment c: the normalised output when the
// piece is the whole segment, else the unnormalised partial (o, m, l) at
// piece index cta + b*Hkv + g.
template <int D, bool FP8>
__device__ __forceinline__ void finish_piece(const DecodeParams& p, SegState<D>& s,
                                             const Cursor& c, bool whole, int32_t cta) {
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  float l0 = s.l[0], l1 = s.l[1];
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  const int h0 = 2 * tq, h1 = 2 * tq + 1;
  if (whole && p.pf_o != nullptr) {
    // cascade: fold in the prefix partial of each head,
    // out = (2^(m-M) acc + 2^(mp-M) op) / (2^(m-M) l + 2^(mp-M) lp)
    const int64_t row = static_cast<int64_t>(c.b) * p.num_q_heads + c.g * p.group;
    __nv_bfloat16* ob = p.out + row * D;
    float a[2] = {0.f, 0.f}, ap[2] = {0.f, 0.f}, inv[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int h = k ? h1 : h0;
      if (h < p.group) {
        const float2 pml = p.pf_ml[row + h];
        const float M = fmaxf(s.m[k], pml.x);
        a[k] = fast_exp2(s.m[k] - M);
        ap[k] = fast_exp2(pml.x - M);
        inv[k] = 1.f / fmaf(k ? l1 : l0, a[k], pml.y * ap[k]);
      }
    }
    // fold the prefix in with loads only (kept in flight together; a store
    // between them would serialise them), then store
#pragma unroll
    for (int i = 0; i < D / 16; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int k = q & 1, h = k ? h1 : h0;
        if (h < p.group)
          s.acc[i][q] = fmaf(s.acc[i][q], a[k],
                             p.pf_o[(row + h) * D + acc_d<D, FP8>(i, q, gq)] * ap[k]);
      }
#pragma unroll
    for (int i = 0; i < D / 16; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int k = q & 1, h = k ? h1 : h0;
        if (h < p.group)
          ob[h * D + acc_d<D, FP8>(i, q, gq)] = __float2bfloat16_rn(s.acc[i][q] * inv[k]);
      }
  } else if (whole) {
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
}

// The math warp: every tile of [lo, hi), segment by segment.  Single-warp
// CTAs (kFused) refill the ring themselves after each tile; two-warp CTAs
// release stages and query slots to the copy warp.  Returns the tiles and
// query slots consumed.
template <int D, bool FP8, bool kFused, bool kAppend = true>
__device__ __forceinline__ void run_math(const DecodeParams& p, const Maps& tm, const Bufs& sb,
                                         Loader& ld, Cursor c, int64_t U, int32_t P,
                                         int64_t lo, int64_t hi, int32_t cta, uint32_t& used,
                                         uint32_t& qread) {
  using L = Smem<D, FP8>;
  Header* hdr = sb.hdr;
  const int lane = threadIdx.x & 31;
  int64_t u = lo;
  used = qread = 0;
  bool ok = true;
  SegState<D> s;
  uint32_t qb[D / 16][2];
  float hm0, hm1;
  if (kFused) top_up<D, FP8, kAppend>(p, tm, sb, ld, hi, used, qread);
  if (p.stall) {  // test hook: a wait that can only run out
    ok = mbar_wait(smem_addr(&hdr->stall), 0, p.wait_limit);
    ok = __all_sync(0xffffffffu, ok);
  }
  while (u < hi && ok) {
    const int32_t seg_end = static_cast<int32_t>(
        min(static_cast<int64_t>(c.T), c.tile + (hi - u)));
    const bool whole = c.tile == 0 && seg_end == c.T;
    const uint32_t qs = qread % kQSlots;
    ok = mbar_wait(smem_addr(&hdr->qfull[qs]), (qread / kQSlots) & 1, p.wait_limit);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    load_query<D, FP8>(p, sb.q + qs * L::kQBytes, qb, hm0, hm1);
    ++qread;
    __syncwarp();
    if (kFused) {
      top_up<D, FP8, kAppend>(p, tm, sb, ld, hi, used, qread);
    } else if (lane == 0) {
      mbar_arrive(smem_addr(&hdr->qempty[qs]));
    }
    seg_reset(s);
    for (int32_t tile = c.tile; tile < seg_end; ++tile) {
      const uint32_t stage = used % p.stages;
      ok = mbar_wait(smem_addr(&hdr->full[stage]), (used / p.stages) & 1, p.wait_limit);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const uint32_t kb = sb.ring + stage * L::kStageBytes;
      const uint32_t vb = kb + L::kKVBytes;
      const int valid = min(kTile, c.n - (p.skip + tile * kTile));
      if (valid < kTile) {
        // Rows past the sequence end hold stale or foreign data: zero the V
        // rows (0 * NaN would poison the MMA); K rows are masked by -inf.
        // The proxy fence orders these writes before the stage's next copy.
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
      ++used;
      __syncwarp();
      if (kFused) {
        top_up<D, FP8, kAppend>(p, tm, sb, ld, hi, used, qread);
      } else if (lane == 0) {
        mbar_arrive(smem_addr(&hdr->empty[stage]));
      }
    }
    if (!ok) break;
    finish_piece<D, FP8>(p, s, c, whole, cta);
    // The CTA that finishes a split segment hands its merge to the merge
    // kernel's CTA of the same index (at most one per CTA: only the first
    // segment of a range can have started in an earlier CTA).
    if (!whole && seg_end == c.T && lane == 0)
      p.ws_job[cta] =
          make_int2(c.b * p.num_kv_heads + c.g, first_cta(p, U, P, u - c.tile, c.b, c.g));
    u += seg_end - c.tile;
    if (u < hi) next_segment(p, c);
  }
}

// ------------------------------------------------------------- kernels ---
// Kernel shape per instantiation, from measurement: bf16 tiles stream at
// the HBM rate when a copy warp sits beside each math warp (the TMA issue
// stalls land on the copy warp); FP8's heavier math wants every warp
// computing, so its CTAs are single warps that issue their own copies.
template <int D, bool FP8>
struct DecodeShape {
  static constexpr bool kTwoWarps = !FP8;
  static constexpr int kThreads = kTwoWarps ? 64 : 32;
};

// Shared-memory carve-up; false if the window is not 1024-aligned (the
// swizzled TMA boxes need it) or the ring depth is out of range.
template <int D, bool FP8>
__device__ __forceinline__ bool carve(const DecodeParams& p, uint8_t* smem_raw, Bufs& sb) {
  using L = Smem<D, FP8>;
  const uint32_t base = smem_addr(smem_raw);
  if ((base & 1023u) || p.stages < 1 || p.stages > kMaxStages) {
    if (threadIdx.x == 0) flag_error(PA_DEVERR_LAUNCH);
    return false;
  }
  sb.q = base;
  sb.ring = base + kQSlots * L::kQBytes;
  sb.hdr = reinterpret_cast<Header*>(smem_raw + kQSlots * L::kQBytes + p.stages * L::kStageBytes);
  return true;
}

// The CTA's work split, before the programmatic-dependency wait: it reads
// only seq_lens, which no kernel of this library writes, so it overlaps
// the tail of the grid before.  After the wait the math warp's lane 0
// clears the CTA's merge job (the previous merge grid may still read the
// job words until then).
__device__ __forceinline__ bool split_then_wait(const DecodeParams& p, int64_t& U, int32_t& P,
                                                int64_t& lo, int64_t& hi, Loader& ld) {
  Cursor c;
  const bool mine = my_range(p, U, P, lo, hi, c);
  if (mine) loader_init(lo, hi, c, ld);
  pdl_wait();
  pdl_trigger();
  if (p.ws_job != nullptr && threadIdx.x == blockDim.x - 32)
    p.ws_job[blockIdx.x] = make_int2(-1, -1);
  return mine;
}

// Two warps: warp 0 copies, warp 1 computes.
template <int D, bool FP8>
__global__ void __launch_bounds__(64, 8)
    paged_decode_ws_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Bufs sb;
  if (!carve<D, FP8>(p, smem_raw, sb)) return;
  const Maps tm{&tm_q, &tm_k, &tm_v};
  if (threadIdx.x == 0) {
    for (int st = 0; st < p.stages; ++st) {
      mbar_init(smem_addr(&sb.hdr->full[st]), 1);
      mbar_init(smem_addr(&sb.hdr->empty[st]), 1);
    }
    for (int st = 0; st < kQSlots; ++st) {
      mbar_init(smem_addr(&sb.hdr->qfull[st]), 1);
      mbar_init(smem_addr(&sb.hdr->qempty[st]), 1);
    }
    mbar_init(smem_addr(&sb.hdr->stall), 1);
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncthreads();
  // Launched as a programmatic dependent: only the work split runs before
  // the wait for the previous grid.
  int64_t U, lo, hi;
  int32_t P;
  Loader ld;
  if (!split_then_wait(p, U, P, lo, hi, ld)) return;
  if (threadIdx.x < 32) {
    produce<D, FP8>(p, tm, sb, ld, hi);
  } else {
    uint32_t used, qread;
    run_math<D, FP8, false>(p, tm, sb, ld, ld.c, U, P, lo, hi, blockIdx.x, used, qread);
  }
}

// One warp that issues its own copies between tiles.  kAppend: compiled
// with the fused FP8 append (a separate instantiation, so that plain
// decode keeps its registers).
template <int D, bool FP8, bool kAppend = false>
__global__ void __launch_bounds__(32, 16)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const DecodeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Bufs sb;
  if (!carve<D, FP8>(p, smem_raw, sb)) return;
  const Maps tm{&tm_q, &tm_k, &tm_v};
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    for (int st = 0; st < p.stages; ++st) mbar_init(smem_addr(&sb.hdr->full[st]), 1);
    for (int st = 0; st < kQSlots; ++st) mbar_init(smem_addr(&sb.hdr->qfull[st]), 1);
    mbar_init(smem_addr(&sb.hdr->stall), 1);
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncwarp();
  int64_t U, lo, hi;  // as in the two-warp kernel
  int32_t P;
  Loader ld;
  if (!split_then_wait(p, U, P, lo, hi, ld)) return;
  uint32_t used, qread;
  run_math<D, FP8, true, kAppend || !FP8>(p, tm, sb, ld, ld.c, U, P, lo, hi, blockIdx.x, used,
                                           qread);
  // No copy may still target shared memory when the CTA exits.  On the
  // normal path every issued copy has been waited for already.
  if (lane == 0) {
    const uint32_t S = p.stages;
    for (uint32_t k = used; k < ld.it; ++k)
      mbar_wait(smem_addr(&sb.hdr->full[k % S]), (k / S) & 1, 1u << 16);
    for (uint32_t k = qread; k < ld.qn; ++k)
      mbar_wait(smem_addr(&sb.hdr->qfull[k % kQSlots]), (k / kQSlots) & 1, 1u << 16);
  }
}

// ----------------------------------------------------------------- merge --
// Launched with one CTA per decode CTA, G * D / 4 threads each.  Writes the sequences the decode
// grid had no tile of (one thread per sequence): zeros for empty ones, the
// normalised prefix partial for a cascade sequence that ends at the prefix.
// Then CTA c merges the split segment decode CTA c finished, if any: thread
// (h, d4) owns 4 output columns of head h, and over the segment's pieces j
// (plus, in a cascade, the prefix partial)
//   M = max_j m_j,  out = sum_j 2^(m_j - M) o_j / sum_j 2^(m_j - M) l_j.
// The loads over pieces are independent, so several are kept in flight.
template <int D>
__global__ void __launch_bounds__(kMaxG * D / 4, 1)
    paged_decode_merge_kernel(const DecodeParams p) {
  pdl_wait();  // the decode grid's partials are complete and visible
  for (int32_t bb = blockIdx.x * blockDim.x + threadIdx.x; bb < p.num_seqs;
       bb += gridDim.x * blockDim.x) {
    const int32_t n = clamp_len(p, p.seq_lens[bb]);
    if (n > p.skip) continue;  // the decode grid covered it
    const int64_t row = static_cast<int64_t>(bb) * p.num_q_heads;
    if (p.pf_o != nullptr && n == p.skip) {
      // cascade, nothing past the prefix: the prefix partial alone
      for (int h = 0; h < p.num_q_heads; ++h) {
        const float inv = 1.f / p.pf_ml[row + h].y;
        for (int d = 0; d < D; ++d)
          p.out[(row + h) * D + d] = __float2bfloat16_rn(p.pf_o[(row + h) * D + d] * inv);
      }
      continue;
    }
    // empty sequence (or, in a cascade, one shorter than the prefix): zeros
    if (n > 0) flag_error(PA_DEVERR_BAD_SEQ_LEN);
    // a fused append needs the new token inside the sequence
    if (p.slot_mapping != nullptr && p.slot_mapping[bb] >= 0) flag_error(PA_DEVERR_BAD_SLOT);
    uint4* o = reinterpret_cast<uint4*>(p.out + row * D);
    for (int i = 0; i < p.num_q_heads * D / 8; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (p.ws_job == nullptr) return;
  const int2 job = p.ws_job[blockIdx.x];
  if (job.x < 0) return;
  const int32_t seg = job.x, c0 = job.y, c1 = blockIdx.x;
  const int32_t b = seg / p.num_kv_heads, g = seg % p.num_kv_heads;
  const int h = threadIdx.x / (D / 4);
  const int d4 = (threadIdx.x % (D / 4)) * 4;
  if (h >= p.group) return;
  __nv_bfloat16* ob = p.out + (static_cast<int64_t>(b) * p.num_q_heads + g * p.group) * D;
  const int np = c1 - c0 + 1;
  const int64_t first = static_cast<int64_t>(seg) + c0;  // piece index of c0
  const float2* ml = p.ws_ml + first * kMaxG + h;
  const float4* o = reinterpret_cast<const float4*>(p.ws_o + (first * kMaxG + h) * D + d4);
  constexpr int kOStride = kMaxG * D / 4;  // float4s per piece
  // (m, l) and rows of up to kBatch pieces are loaded together, so a job
  // costs one round trip after its job word rather than two
  constexpr int kBatch = 8;
  float2 v[kBatch];
  float4 x[kBatch];
#pragma unroll
  for (int k = 0; k < kBatch; ++k)
    if (k < np) {
      v[k] = ml[k * kMaxG];
      x[k] = o[k * kOStride];
    }
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kBatch; ++k)
    if (k < np) M = fmaxf(M, v[k].x);
  for (int k = kBatch; k < np; ++k) M = fmaxf(M, ml[k * kMaxG].x);
  float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (p.pf_o != nullptr) {
    // cascade: the prefix partial is one more piece
    const int64_t row = static_cast<int64_t>(b) * p.num_q_heads + g * p.group + h;
    const float2 pml = p.pf_ml[row];
    const float4 y = *reinterpret_cast<const float4*>(p.pf_o + row * D + d4);
    M = fmaxf(M, pml.x);
    const float w = fast_exp2(pml.x - M);
    num = make_float4(w * y.x, w * y.y, w * y.z, w * y.w);
    den = w * pml.y;
  }
#pragma unroll
  for (int k = 0; k < kBatch; ++k)
    if (k < np) {
      const float w = fast_exp2(v[k].x - M);
      num.x = fmaf(w, x[k].x, num.x);
      num.y = fmaf(w, x[k].y, num.y);
      num.z = fmaf(w, x[k].z, num.z);
      num.w = fmaf(w, x[k].w, num.w);
      den = fmaf(w, v[k].y, den);
    }
#pragma unroll 4
  for (int k = kBatch; k < np; ++k) {
    const float2 vv = ml[k * kMaxG];
    const float4 xx = o[k * kOStride];
    const float w = fast_exp2(vv.x - M);
    num.x = fmaf(w, xx.x, num.x);
    num.y = fmaf(w, xx.y, num.y);
    num.z = fmaf(w, xx.z, num.z);
    num.w = fmaf(w, xx.w, num.w);
    den = fmaf(w, vv.y, den);
  }
  uint2 r;
  r.x = pack_bf16x2(num.x / den, num.y / den);
  r.y = pack_bf16x2(num.z / den, num.w / den);
  *reinterpret_cast<uint2*>(ob + h * D + d4) = r;
}

}  // namespace pa
