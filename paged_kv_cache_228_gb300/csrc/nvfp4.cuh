// NVFP4 KV cache: quantised append and paged decode for sm_103a.
//
// "Paged Attention and KV Cache Fragmentation", section "Quantization as a
// way to stretch paged memory further": NVFP4, the Blackwell-only cache
// format, halves FP8's footprint again.  The pages do not define it; this
// is NVIDIA's published NVFP4: FP4 E2M1 values (OCP MX element format), one
// E4M3 scale per 16 consecutive values of a head row, and one fp32 scale S
// per tensor (the K, resp. V, cache of a layer) supplied by the caller.
//
//   block scale   s_g = e4m3_rne_sat(max|x_g| / (6 S))
//   value         q_i = e2m1_rne_sat(x_i / (e4m3(s_g) S))   (0 when s_g = 0)
//   decoded       x_i ~ e2m1(q_i) * e4m3(s_g) * S
//
// every division and product of the encoder in IEEE fp32.
//
// Layout per (block, KV head), chosen so that each lane of the decode warp
// loads exactly the bytes of its MMA fragments with one 16-byte copy per row
// (8 bytes at D = 64):
//   k     [bs][D/2]      two values of a token per byte, even d low nibble
//   k_sf  [bs][D/16]     E4M3 scale of each 16-value group of a token
//   v     [bs/2][D]      "pair-rows": byte d holds tokens 2p (low nibble) and
//                        2p + 1 (high nibble) of dimension d
//   v_sf  [D/16][bs]     E4M3 scale per (group, token), group-major
//
// Decode work split, partials and merge are the bf16/FP8 kernels' (flat
// 16-token tiles over persistent CTAs, log-sum-exp merge).  A tile's bytes
// go to shared memory with per-lane cp.async into a ring of kStages stages
// (each lane copies what it will read itself; the scale bytes are copied
// by D/8 lanes and read after a warp barrier), two tiles per loop step
// while two remain.  Math on the f16 tensor-core
// MMA, fp32 accumulate, in the same fragment layout as the other kernels
// (tokens on M, the query heads of the group on N):
//   S^T = K' . Q^T with K' = e2m1 * e4m3 block scale, formed exactly in f16
//         registers from the packed bytes (at most 6 significant bits and
//         at most 6 * 448 in magnitude); a permutation of d shared by K' and
//         Q lets lane (gq, tq) take d in [2 (D/8) tq, 2 (D/8) (tq + 1)),
//         so its K bytes are contiguous;
//   O^T += V'^T . P^T with V' from the pair-rows, again exact in f16; lane gq
//         owns d in [(D/8) gq, (D/8)(gq + 1)) of every m-tile, one group.
// The tensor scales fold in after the MMA: S_k into the score multiplier,
// S_v into the final normalisation.  A second instantiation fuses the
// step's append: the warp that copies a segment's last tile first writes
// that head's new rows into it (fp4_append_new).
#pragma once

#include "decode.cuh"

namespace pa {

struct Fp4Args {
  const __nv_bfloat16* q;  // [B][Hq][D]
  uint8_t* k;              // pools; written only by the fused append
  uint8_t* v;
  uint8_t* k_sf;
  uint8_t* v_sf;
  float k_gs, v_gs;  // tensor scales S_k, S_v
  // Fused append (null when off): sequence b's new token rows
  // k_new/v_new[b][Hkv][D] go to slot_mapping[b] (< 0: none), which must be
  // the slot the table gives position seq_lens[b] - 1.
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int64_t* slot_mapping;
};

template <int D>
struct Fp4Layout {
  static constexpr int kTB = D / 8;                    // bytes a lane owns of a row
  static constexpr int kK = 0;                         // K: 16 rows x D/2
  static constexpr int kV = kTile * D / 2;             // V: 8 pair-rows x D
  static constexpr int kKsf = kV + kTile / 2 * D;      // 16 tokens x D/16
  static constexpr int kVsf = kKsf + D;                // D/16 groups x 16 tokens
  static constexpr int kStage = kVsf + D;
  static constexpr int kStages = D == 128 ? 5 : 8;
  static_assert(kStage % 128 == 0, "stage alignment");
};

template <int D>
constexpr size_t fp4_smem_bytes() {
  return static_cast<size_t>(Fp4Layout<D>::kStages) * Fp4Layout<D>::kStage;
}

// N-byte async copy global -> shared (N = 16: L2 only; 4 or 8: through L1);
// ok = false writes N zero bytes and reads nothing.
template <int N>
__device__ __forceinline__ void fp4_cp_async(uint32_t dst, const void* src, bool ok) {
  if constexpr (N == 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(ok ? 16 : 0)
                 : "memory");
  } else {
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(dst), "l"(src), "n"(N),
                 "r"(ok ? N : 0)
                 : "memory");
  }
}

__device__ __forceinline__ void fp4_cp_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void fp4_cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Four bytes of E2M1 pairs -> four f16x2 (byte k: low nibble -> low half,
// high nibble -> high half).  Exact: every E2M1 value is an f16 value.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& d0, uint32_t& d1,
                                                uint32_t& d2, uint32_t& d3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
      : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// E2M1 code of y, round to nearest with ties to the even code, saturating
// to +-6; NaN -> +6.  Thresholds are the midpoints of the grid 0, .5, 1,
// 1.5, 2, 3, 4, 6: a tie stays on the lower neighbour when that neighbour's
// mantissa bit is 0 (">"), moves up when it is 1 (">=").
__device__ __forceinline__ uint32_t e2m1_rne(float y) {
  const float a = fabsf(y);
  const uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                     (a >= 3.5f) + (a > 5.f);
  if (a != a) return 7u;
  return c | (signbit(y) ? 8u : 0u);
}

// Byte offset of lane-chunk c (D/8 bytes) of pair-row r in a stage's V
// area, XOR-swizzled so that the 8 (D = 128: 16-byte loads) or 16 (D = 64:
// 8-byte loads) lanes of one shared-memory phase hit distinct banks.
template <int D>
__device__ __forceinline__ uint32_t fp4_vchunk(int r, int c) {
  if (D == 128) return r * 128 + ((c ^ (2 * (r & 3))) << 4);
  return r * 64 + ((c ^ (4 * ((r >> 1) & 1))) << 3);
}

template <int N>
__device__ __forceinline__ void lds_words(uint32_t addr, uint32_t (&w)[N / 4]) {
  if constexpr (N == 16) {
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(addr));
  } else {
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(addr));
  }
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// f16x2 (s, s) of the E4M3 scale byte b.
__device__ __forceinline__ uint32_t sf_splat(uint32_t b) {
  return e4m3x2_to_f16x2(static_cast<uint16_t>(b * 0x0101u));
}

// Table entry of the block holding tile c.tile of segment c.
__device__ __forceinline__ int32_t fp4_entry(const DecodeParams& p, const Cursor& c) {
  return p.block_tables[static_cast<int64_t>(c.b) * p.max_blocks +
                        ((c.tile * kTile) >> p.log2_bs)];
}

// Copy tile c (in block blk) into the stage at st.  An id outside the pool
// fills the stage with zeros and flags PA_DEVERR_BAD_BLOCK_ID.
template <int D>
__device__ __forceinline__ void fp4_issue(const DecodeParams& p, const Fp4Args& f, uint32_t st,
                                          const Cursor& c, int32_t blk) {
  using L = Fp4Layout<D>;
  constexpr int TB = L::kTB, NG = D / 16;
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  const bool ok = blk >= 0 && blk < p.num_blocks;
  if (!ok && lane == 0) flag_error(PA_DEVERR_BAD_BLOCK_ID);
  const int32_t off = (c.tile * kTile) & (p.block_size - 1);
  const int64_t hb = ok ? static_cast<int64_t>(blk) * p.num_kv_heads + c.g : 0;
  const int64_t row0 = hb * p.block_size + off;  // first token row of the tile
  const uint8_t* kr = f.k + row0 * (D / 2) + TB * tq;
  fp4_cp_async<TB>(st + L::kK + gq * (D / 2) + TB * tq, kr + gq * (D / 2), ok);
  fp4_cp_async<TB>(st + L::kK + (gq + 8) * (D / 2) + TB * tq, kr + (gq + 8) * (D / 2), ok);
  const uint8_t* vr = f.v + (hb * (p.block_size >> 1) + (off >> 1)) * D + TB * gq;
  fp4_cp_async<TB>(st + L::kV + fp4_vchunk<D>(tq, gq), vr + tq * D, ok);
  fp4_cp_async<TB>(st + L::kV + fp4_vchunk<D>(tq + 4, gq), vr + (tq + 4) * D, ok);
  if (lane < NG)
    fp4_cp_async<16>(st + L::kKsf + 16 * lane, f.k_sf + row0 * NG + 16 * lane, ok);
  else if (lane < 2 * NG)
    fp4_cp_async<16>(st + L::kVsf + 16 * (lane - NG),
                     f.v_sf + (hb * NG + (lane - NG)) * p.block_size + off, ok);
}

// Query fragments of segment c (B operand: n = head gq, k = the permuted
// d): qf[j][0] = q[gq][2TB tq + 4j + {0, 1}], qf[j][1] = ... + {2, 3}, in
// f16 (heads past the group are zeros).
template <int D>
__device__ __forceinline__ void fp4_load_query(const DecodeParams& p, const Fp4Args& f,
                                               const Cursor& c, uint32_t (&qf)[D / 16][2]) {
  constexpr int TB = D / 8;
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  if (gq >= p.group) {
#pragma unroll
    for (int j = 0; j < D / 16; ++j) qf[j][0] = qf[j][1] = 0u;
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(
      f.q + (static_cast<int64_t>(c.b) * p.num_q_heads + c.g * p.group + gq) * D + 2 * TB * tq);
#pragma unroll
  for (int u = 0; u < TB / 4; ++u) {  // 8 values per load
    const uint4 w = __ldg(src + u);
    const float2 e0 = unpack_bf16x2(w.x), e1 = unpack_bf16x2(w.y);
    const float2 e2 = unpack_bf16x2(w.z), e3 = unpack_bf16x2(w.w);
    qf[2 * u][0] = pack_f16x2(e0.x, e0.y);
    qf[2 * u][1] = pack_f16x2(e1.x, e1.y);
    qf[2 * u + 1][0] = pack_f16x2(e2.x, e2.y);
    qf[2 * u + 1][1] = pack_f16x2(e3.x, e3.y);
  }
}

// Masked scores (log2 units) of one tile: x = (row gq, head 2tq), (gq, 2tq+1),
// (gq+8, 2tq), (gq+8, 2tq+1).
template <int D>
__device__ __forceinline__ void fp4_qk(uint32_t st, int valid, const uint32_t (&qf)[D / 16][2],
                                       float kmul, float (&x)[4]) {
  using L = Fp4Layout<D>;
  constexpr int TB = L::kTB;
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  // K rows gq and gq + 8, the lane's TB bytes; their block scales
  uint32_t k0[TB / 4], k1[TB / 4];
  lds_words<TB>(st + L::kK + gq * (D / 2) + TB * tq, k0);
  lds_words<TB>(st + L::kK + (gq + 8) * (D / 2) + TB * tq, k1);
  uint32_t s0[2], s1[2];
  if (D == 128) {  // groups 2tq, 2tq + 1
    const uint32_t p0 = e4m3x2_to_f16x2(static_cast<uint16_t>(lds_u16(st + L::kKsf + gq * 8 + 2 * tq)));
    const uint32_t p1 =
        e4m3x2_to_f16x2(static_cast<uint16_t>(lds_u16(st + L::kKsf + (gq + 8) * 8 + 2 * tq)));
    s0[0] = __byte_perm(p0, 0, 0x1010);
    s0[1] = __byte_perm(p0, 0, 0x3232);
    s1[0] = __byte_perm(p1, 0, 0x1010);
    s1[1] = __byte_perm(p1, 0, 0x3232);
  } else {  // group tq
    s0[0] = s0[1] = sf_splat(lds_u8(st + L::kKsf + gq * 4 + tq));
    s1[0] = s1[1] = sf_splat(lds_u8(st + L::kKsf + (gq + 8) * 4 + tq));
  }
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int w = 0; w < TB / 4; ++w) {  // word w: bytes 4w..4w+3, k-steps 2w, 2w + 1
    uint32_t r0[4], r1[4];
    e2m1x8_to_f16x2(k0[w], r0[0], r0[1], r0[2], r0[3]);
    e2m1x8_to_f16x2(k1[w], r1[0], r1[1], r1[2], r1[3]);
    const int hsel = (D == 128) ? (w >> 1) : 0;  // group 2tq + (j >= 4)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = 2 * w + h;
      const uint32_t a0 = hmul2_u32(r0[2 * h], s0[hsel]);
      const uint32_t a1 = hmul2_u32(r1[2 * h], s1[hsel]);
      const uint32_t a2 = hmul2_u32(r0[2 * h + 1], s0[hsel]);
      const uint32_t a3 = hmul2_u32(r1[2 * h + 1], s1[hsel]);
      if (h)
        mma_f16(sb, a0, a1, a2, a3, qf[j][0], qf[j][1]);
      else
        mma_f16(sa, a0, a1, a2, a3, qf[j][0], qf[j][1]);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) x[q] = (sa[q] + sb[q]) * kmul;
  if (valid < kTile) {  // the segment's last tile (warp-uniform)
    if (gq >= valid) x[0] = x[1] = -INFINITY;
    if (gq + 8 >= valid) x[2] = x[3] = -INFINITY;
  }
}

// O^T += V'^T . P^T for one tile.  V pair-rows tq (tokens 2tq, 2tq+1) and
// tq + 4 (2tq+8, 2tq+9); the scales of those tokens in the lane's group are
// zeroed past the sequence end (those slots may hold anything, and P = 0
// must meet finite V).
template <int D>
__device__ __forceinline__ void fp4_pv(uint32_t st, int valid, uint32_t pb0, uint32_t pb1,
                                       SegState<D>& s) {
  using L = Fp4Layout<D>;
  constexpr int TB = L::kTB;
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  uint32_t v0[TB / 4], v1[TB / 4];
  lds_words<TB>(st + L::kV + fp4_vchunk<D>(tq, gq), v0);
  lds_words<TB>(st + L::kV + fp4_vchunk<D>(tq + 4, gq), v1);
  const int gv = D == 128 ? gq : (gq >> 1);
  uint32_t wa = lds_u16(st + L::kVsf + gv * 16 + 2 * tq);
  uint32_t wb = lds_u16(st + L::kVsf + gv * 16 + 2 * tq + 8);
  if (valid < kTile) {
    if (2 * tq >= valid) wa &= 0xff00u;
    if (2 * tq + 1 >= valid) wa &= 0x00ffu;
    if (2 * tq + 8 >= valid) wb &= 0xff00u;
    if (2 * tq + 9 >= valid) wb &= 0x00ffu;
  }
  const uint32_t sA = e4m3x2_to_f16x2(static_cast<uint16_t>(wa));
  const uint32_t sB = e4m3x2_to_f16x2(static_cast<uint16_t>(wb));
#pragma unroll
  for (int w = 0; w < TB / 8; ++w) {  // m-tiles 4w..4w+3: bytes 4w+b and TB/2 + 4w + b
    uint32_t lo0[4], hi0[4], lo1[4], hi1[4];
    e2m1x8_to_f16x2(v0[w], lo0[0], lo0[1], lo0[2], lo0[3]);
    e2m1x8_to_f16x2(v0[w + TB / 8], hi0[0], hi0[1], hi0[2], hi0[3]);
    e2m1x8_to_f16x2(v1[w], lo1[0], lo1[1], lo1[2], lo1[3]);
    e2m1x8_to_f16x2(v1[w + TB / 8], hi1[0], hi1[1], hi1[2], hi1[3]);
#pragma unroll
    for (int b = 0; b < 4; ++b)
      mma_f16(s.acc[4 * w + b], hmul2_u32(lo0[b], sA), hmul2_u32(hi0[b], sA),
              hmul2_u32(lo1[b], sB), hmul2_u32(hi1[b], sB), pb0, pb1);
  }
}

// One tile: scores, online softmax, O^T update.
template <int D>
__device__ __forceinline__ void fp4_tile(uint32_t st, int valid, const uint32_t (&qf)[D / 16][2],
                                         float kmul, SegState<D>& s) {
  float x[4];
  fp4_qk<D>(st, valid, qf, kmul, x);
  float alpha0, alpha1;
  uint32_t pb0, pb1;
  softmax_tile<true>(x[0], x[1], x[2], x[3], s.m, s.l, 1.f, 1.f, alpha0, alpha1, pb0, pb1);
  rescale(s, alpha0, alpha1);
  fp4_pv<D>(st, valid, pb0, pb1, s);
}

// Two consecutive tiles of one segment (the first one full): both score
// blocks, one online-softmax update over their 32 tokens (the running max
// moves only when a score passes it by more than 8 in log2 units, as in
// softmax_tile), then both O^T updates.
template <int D>
__device__ __forceinline__ void fp4_tile2(uint32_t sta, uint32_t stb, int valid_b,
                                          const uint32_t (&qf)[D / 16][2], float kmul,
                                          SegState<D>& s) {
  float xa[4], xb[4];
  fp4_qk<D>(sta, kTile, qf, kmul, xa);
  fp4_qk<D>(stb, valid_b, qf, kmul, xb);
  constexpr float kSlack = 8.f;
  float mx0 = fmaxf(fmaxf(xa[0], xa[2]), fmaxf(xb[0], xb[2]));
  float mx1 = fmaxf(fmaxf(xa[1], xa[3]), fmaxf(xb[1], xb[3]));
  float alpha0 = 1.f, alpha1 = 1.f;
  if (__any_sync(0xffffffffu, mx0 > s.m[0] + kSlack || mx1 > s.m[1] + kSlack)) {
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
  rescale(s, alpha0, alpha1);
  fp4_pv<D>(sta, kTile, movmatrix_t(pack_f16x2(pa[0], pa[1])),
            movmatrix_t(pack_f16x2(pa[2], pa[3])), s);
  fp4_pv<D>(stb, valid_b, movmatrix_t(pack_f16x2(pb[0], pb[1])),
            movmatrix_t(pack_f16x2(pb[2], pb[3])), s);
}

// Write a finished piece (as finish_piece: the output when the piece is the
// whole segment, else the partial at piece cta + b*Hkv + g).  Accumulator
// (i, q) of lane (gq, tq) is d = TB gq + i + (q >> 1) TB/2, head 2tq + (q & 1).
template <int D>
__device__ __forceinline__ void fp4_finish(const DecodeParams& p, const Fp4Args& f,
                                           SegState<D>& s, const Cursor& c, bool whole,
                                           int32_t cta) {
  constexpr int TB = D / 8;
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  float l[2] = {s.l[0], s.l[1]};
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l[0] += __shfl_xor_sync(0xffffffffu, l[0], o);
    l[1] += __shfl_xor_sync(0xffffffffu, l[1], o);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int h = 2 * tq + k;
    if (h >= p.group) continue;
    float v[TB];
#pragma unroll
    for (int i = 0; i < TB / 2; ++i) {
      v[i] = s.acc[i][k];
      v[i + TB / 2] = s.acc[i][k + 2];
    }
    if (whole) {
      const float sc = f.v_gs / l[k];
      __nv_bfloat16* ob = p.out + (static_cast<int64_t>(c.b) * p.num_q_heads + c.g * p.group + h) * D +
                          TB * gq;
#pragma unroll
      for (int u = 0; u < TB / 8; ++u) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * u] * sc, v[8 * u + 1] * sc);
        w.y = pack_bf16x2(v[8 * u + 2] * sc, v[8 * u + 3] * sc);
        w.z = pack_bf16x2(v[8 * u + 4] * sc, v[8 * u + 5] * sc);
        w.w = pack_bf16x2(v[8 * u + 6] * sc, v[8 * u + 7] * sc);
        reinterpret_cast<uint4*>(ob)[u] = w;
      }
    } else {
      const int64_t piece = static_cast<int64_t>(cta) + c.b * p.num_kv_heads + c.g;
      float4* wo = reinterpret_cast<float4*>(p.ws_o + (piece * kMaxG + h) * D + TB * gq);
#pragma unroll
      for (int u = 0; u < TB / 4; ++u)
        wo[u] = make_float4(v[4 * u] * f.v_gs, v[4 * u + 1] * f.v_gs, v[4 * u + 2] * f.v_gs,
                            v[4 * u + 3] * f.v_gs);
      if (gq == 0) p.ws_ml[piece * kMaxG + h] = make_float2(s.m[k], l[k]);
    }
  }
}

// ------------------------------------------------------------ row writer --
// Quantise one bf16 row x (D values) with tensor scale gs into token `off`
// of (block, KV head) hb: the K layout (kv = 0) or the V layout (kv = 1).
// Warp-collective: lane l quantises values [E l, E l + E), E = D / 32, with
// the lanes of its 16-value group.  A V value is one nibble of its
// pair-row byte, which the token's neighbour shares, so V bytes are updated
// by word atomics on disjoint nibbles.
template <int D>
__device__ __forceinline__ void fp4_put_row(const __nv_bfloat16* __restrict__ x, int kv, float gs,
                                            int64_t hb, int64_t off, int32_t block_size,
                                            uint8_t* k, uint8_t* k_sf, uint8_t* v,
                                            uint8_t* v_sf) {
  constexpr int E = D / 32;    // values per lane
  constexpr int LPG = 16 / E;  // lanes per group
  constexpr int NG = D / 16;
  const int lane = threadIdx.x & 31;
  float xv[E];
  if constexpr (E == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(x + E * lane);
    const float2 a = unpack_bf16x2(w.x), b = unpack_bf16x2(w.y);
    xv[0] = a.x; xv[1] = a.y; xv[2] = b.x; xv[3] = b.y;
  } else {
    const float2 a = unpack_bf16x2(*reinterpret_cast<const uint32_t*>(x + E * lane));
    xv[0] = a.x; xv[1] = a.y;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(xv[i]));
#pragma unroll
  for (int o = 1; o < LPG; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const uint32_t sf = f32x2_to_e4m3x2(__fdiv_rn(amax, __fmul_rn(6.f, gs)), 0.f) & 0xffu;
  const float sv = unpack_f16x2(e4m3x2_to_f16x2(static_cast<uint16_t>(sf))).x;
  uint32_t codes = 0;  // value i of the lane in bits 4i..4i+3
  if (sv > 0.f) {
    const float den = __fmul_rn(sv, gs);
#pragma unroll
    for (int i = 0; i < E; ++i) codes |= e2m1_rne(__fdiv_rn(xv[i], den)) << (4 * i);
  }
  const int grp = lane / LPG;
  if (kv == 0) {
    uint8_t* dst = k + (hb * block_size + off) * (D / 2) + (E / 2) * lane;
    if constexpr (E == 4)
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(codes);
    else
      *dst = static_cast<uint8_t>(codes);
    if (lane % LPG == 0) k_sf[(hb * block_size + off) * NG + grp] = static_cast<uint8_t>(sf);
  } else {
    // bytes E*lane .. E*lane + E - 1 of pair-row off/2, nibble off & 1
    const int nib = static_cast<int>(off & 1) * 4;
    uint32_t val = 0, mask = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      val |= ((codes >> (4 * i)) & 0xFu) << (8 * i + nib);
      mask |= 0xFu << (8 * i + nib);
    }
    uint8_t* row = v + (hb * (block_size >> 1) + (off >> 1)) * D;
    const int byte = E * lane;
    const int shift = (byte & 3) * 8;
    unsigned int* word = reinterpret_cast<unsigned int*>(row + (byte & ~3));
    atomicAnd(word, ~(mask << shift));
    atomicOr(word, val << shift);
    if (lane % LPG == 0) v_sf[(hb * NG + grp) * block_size + off] = static_cast<uint8_t>(sf);
  }
}

// The fused append: before the copy of segment c's last tile (in block
// blk), quantise its sequence's new K and V rows of head c.g into position
// n - 1.  A slot that is not that position's is not written and flags
// PA_DEVERR_BAD_SLOT.  The rows are visible to the warp's copies after the
// block-scope fence and the warp barrier.
template <int D>
__device__ __forceinline__ void fp4_append_new(const DecodeParams& p, const Fp4Args& f,
                                               const Cursor& c, int32_t blk) {
  const int64_t slot = f.slot_mapping[c.b];
  if (slot < 0) return;
  const int64_t off = (c.n - 1) & (p.block_size - 1);
  if (blk < 0 || blk >= p.num_blocks ||
      slot != static_cast<int64_t>(blk) * p.block_size + off) {
    if ((threadIdx.x & 31) == 0) flag_error(PA_DEVERR_BAD_SLOT);
    return;
  }
  const int64_t hb = static_cast<int64_t>(blk) * p.num_kv_heads + c.g;
  const int64_t row = (static_cast<int64_t>(c.b) * p.num_kv_heads + c.g) * D;
  fp4_put_row<D>(f.k_new + row, 0, f.k_gs, hb, off, p.block_size, f.k, f.k_sf, f.v, f.v_sf);
  fp4_put_row<D>(f.v_new + row, 1, f.v_gs, hb, off, p.block_size, f.k, f.k_sf, f.v, f.v_sf);
  __threadfence_block();
  __syncwarp();
}

// One warp per CTA; tiles [lo, hi) of the flat list, kStages - 1 tiles in
// flight ahead of the one computed.  Every cp.async group is waited for
// before the CTA exits.  kAppend: the fused append (a separate
// instantiation, so that plain decode keeps its registers).
template <int D, bool kAppend>
__global__ void __launch_bounds__(32, 16)
    paged_decode_nvfp4_kernel(const DecodeParams p, const Fp4Args f) {
  using L = Fp4Layout<D>;
  constexpr int S = L::kStages;
  extern __shared__ __align__(128) uint8_t fp4_smem[];
  const uint32_t ring = smem_addr(fp4_smem);
  const int lane = threadIdx.x & 31;
  // the work split reads only seq_lens: before the programmatic-dependency
  // wait (as in the other decode kernels); the merge job after it
  int64_t U, lo, hi;
  int32_t P;
  Cursor c;
  const bool mine = my_range(p, U, P, lo, hi, c);
  pdl_wait();
  pdl_trigger();
  if (p.ws_job != nullptr && lane == 0) p.ws_job[blockIdx.x] = make_int2(-1, -1);
  if (!mine) return;
  // load side: cursor lc at flat index lu, its block id prefetched
  Cursor lc = c;
  int64_t lu = lo;
  int32_t lblk = fp4_entry(p, lc);
  int ls = 0;  // stage of tile lu
  auto top_up = [&]() {
    if (lu < hi) {
      if (kAppend && lc.tile == lc.T - 1) fp4_append_new<D>(p, f, lc, lblk);
      fp4_issue<D>(p, f, ring + ls * L::kStage, lc, lblk);
      ls = ls + 1 == S ? 0 : ls + 1;
      if (++lu < hi) {
        if (++lc.tile == lc.T) {
          next_segment(p, lc);
          // its query rows (and new K/V rows) into L1 while the tiles
          // before it are computed
          if ((threadIdx.x >> 2) < p.group)
            asm volatile("prefetch.global.L1 [%0];" ::"l"(
                f.q + (static_cast<int64_t>(lc.b) * p.num_q_heads + lc.g * p.group +
                       (threadIdx.x >> 2)) * D + 2 * (D / 8) * (threadIdx.x & 3)));
          if (kAppend) {
            const int64_t row =
                (static_cast<int64_t>(lc.b) * p.num_kv_heads + lc.g) * D + (D / 32) * lane;
            asm volatile("prefetch.global.L1 [%0];" ::"l"(f.k_new + row));
            asm volatile("prefetch.global.L1 [%0];" ::"l"(f.v_new + row));
          }
        }
        lblk = fp4_entry(p, lc);
      }
    }
    fp4_cp_commit();
  };
#pragma unroll 1
  for (int k = 0; k < S - 1; ++k) top_up();
  const float kmul = f.k_gs * p.scale_log2;
  int cs = 0;  // stage of tile u
  int64_t u = lo;
  SegState<D> s;
  uint32_t qf[D / 16][2];
  while (u < hi) {
    const int32_t seg_end = static_cast<int32_t>(min(static_cast<int64_t>(c.T), c.tile + (hi - u)));
    const bool whole = c.tile == 0 && seg_end == c.T;
    const int64_t useg = u - c.tile;  // flat index of the segment's tile 0
    fp4_load_query<D>(p, f, c, qf);
    seg_reset(s);
#pragma unroll 1
    // Two tiles per step while two remain.  Each step starts with one copy
    // issued; a pair step issues its second copy after both of its stages
    // are read, so kStages - 2 tiles stay in flight during its math.
    for (int32_t tile = c.tile; tile < seg_end;) {
      top_up();
      if (tile + 1 < seg_end) {
        fp4_cp_wait<S - 2>();  // tiles u and u + 1 have landed
        __syncwarp();
        const int cs2 = cs + 1 == S ? 0 : cs + 1;
        fp4_tile2<D>(ring + cs * L::kStage, ring + cs2 * L::kStage,
                     min(kTile, c.n - (tile + 1) * kTile), qf, kmul, s);
        cs = cs2 + 1 == S ? 0 : cs2 + 1;
        __syncwarp();  // both stages are read before later copies overwrite them
        top_up();
        tile += 2;
      } else {
        fp4_cp_wait<S - 1>();  // tile u has landed
        __syncwarp();
        fp4_tile<D>(ring + cs * L::kStage, min(kTile, c.n - tile * kTile), qf, kmul, s);
        cs = cs + 1 == S ? 0 : cs + 1;
        __syncwarp();
        ++tile;
      }
    }
    fp4_finish<D>(p, f, s, c, whole, blockIdx.x);
    if (!whole && seg_end == c.T && lane == 0)
      p.ws_job[blockIdx.x] =
          make_int2(c.b * p.num_kv_heads + c.g, first_cta(p, U, P, useg, c.b, c.g));
    u += seg_end - c.tile;
    if (u < hi) next_segment(p, c);
  }
  fp4_cp_wait<0>();
}

// ------------------------------------------------------------ cache write --
// One warp per (token, K or V, KV head) row (fp4_put_row).
template <int D>
__global__ void __launch_bounds__(256)
    cache_write_nvfp4_kernel(const __nv_bfloat16* __restrict__ k_new,
                             const __nv_bfloat16* __restrict__ v_new,
                             const int64_t* __restrict__ slots, int32_t num_tokens,
                             int32_t num_kv_heads, int32_t block_size, int64_t num_slots,
                             uint8_t* __restrict__ k, uint8_t* __restrict__ k_sf,
                             uint8_t* __restrict__ v, uint8_t* __restrict__ v_sf, float k_gs,
                             float v_gs) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t rows = 2LL * num_tokens * num_kv_heads;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < rows; r += nw) {
    const int32_t h = static_cast<int32_t>(r % num_kv_heads);
    const int kv = static_cast<int>((r / num_kv_heads) & 1);
    const int64_t t = r / (2LL * num_kv_heads);
    const int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (lane == 0 && kv == 0 && h == 0) flag_error(PA_DEVERR_BAD_SLOT);
      continue;
    }
    const int64_t blk = slot / block_size, off = slot - blk * block_size;
    fp4_put_row<D>((kv ? v_new : k_new) + (t * num_kv_heads + h) * D, kv, kv ? v_gs : k_gs,
                   blk * num_kv_heads + h, off, block_size, k, k_sf, v, v_sf);
  }
}

}  // namespace pa
