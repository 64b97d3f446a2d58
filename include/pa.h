/*
 * pa.h -- C ABI of libpa, a paged KV cache and paged decode attention
 * library for NVIDIA GB300 (sm_103a).
 *
 * The method (three web pages on KV cache fragmentation and PagedAttention):
 *   - "KV cache fragmentation" (field guide), section "Definition": the KV
 *     cache is cut into small fixed-size pages; each request owns a logical
 *     sequence of pages that may sit anywhere in physical memory, reached
 *     through a small indirection table, and the attention kernel walks that
 *     table.
 *   - "Paged Attention and KV Cache Fragmentation", section "How
 *     PagedAttention maps an OS concept onto GPU memory": fixed-size blocks
 *     holding a set number of key/value vectors per head; a block table per
 *     request mapping logical positions to physical blocks; blocks allocated
 *     only as a sequence grows and freed when it finishes; requests with a
 *     shared prefix point at the same physical blocks.
 *   - same page, section "Quantization as a way to stretch paged memory
 *     further": FP8 KV caches with full fp32 accumulation, and NVFP4 on
 *     Blackwell.
 *
 * Conventions (all entry points):
 *   - Every function returns a pa_status; nothing throws or aborts.
 *   - Arguments are validated on the host before anything is enqueued; on a
 *     failed check the call returns PA_ERR_INVALID_ARG (or
 *     PA_ERR_UNSUPPORTED for a valid but unimplemented shape) and has no
 *     side effects.
 *   - Device entry points take caller-owned DEVICE pointers, enqueue work on
 *     `stream` (a cudaStream_t passed as void*; NULL = legacy default stream)
 *     and return without synchronising.  A launch failure returns
 *     PA_ERR_CUDA.  Device pointers must be 16-byte aligned.
 *   - Data-dependent errors found on the device (a block id outside the
 *     pool, a slot outside the pool, a sequence longer than its table) never
 *     fault: the offending access is skipped (reads become zeros) and a bit
 *     is set in a per-device error word read by pa_get_device_error().
 *   - The library allocates no device memory in any entry point except that
 *     the CUDA runtime lazily creates its context.  The only host memory it
 *     owns is the opaque pa_allocator.
 *   - Kernels launch as programmatic dependents of the work before them in
 *     the stream and wait for it on the device before touching its data,
 *     with one exception: the decode kernels read seq_lens to split the work
 *     before that wait.  No kernel of this library writes seq_lens; a kernel
 *     of the caller's that produces seq_lens and lets dependents start early
 *     (griddepcontrol.launch_dependents) must not directly precede a decode
 *     call.  Ordinary stream order (copies, kernels without that trigger)
 *     needs nothing.
 *   - Layouts are dense, row-major (last index fastest):
 *       k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *                          bf16 (PA_KV_BF16) or E4M3 bytes (PA_KV_FP8_E4M3)
 *       k_scale, v_scale : float [num_blocks][num_kv_heads] (FP8 only)
 *       block_tables     : int32 [num_seqs][max_blocks_per_seq]; entries at
 *                          or past ceil(seq_len / block_size) are never read
 *                          (pad them with -1)
 *       seq_lens         : int32 [num_seqs], lengths including the token
 *                          appended by this step
 *       q, out           : bf16 [num_seqs][num_q_heads][head_dim]
 *     Query head h reads KV head h / (num_q_heads / num_kv_heads).
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,   /* bad pointer, size, shape or alignment       */
  PA_ERR_OUT_OF_BLOCKS = 2, /* allocator: not enough free blocks           */
  PA_ERR_BAD_BLOCK_ID = 3,  /* allocator: id outside the pool or not live  */
  PA_ERR_CUDA = 4,          /* a CUDA runtime call failed                  */
  PA_ERR_UNSUPPORTED = 5,   /* valid request, shape not implemented        */
  PA_ERR_WORKSPACE = 6      /* workspace missing or smaller than required  */
} pa_status;

typedef enum pa_kv_dtype {
  PA_KV_BF16 = 0,
  PA_KV_FP8_E4M3 = 1,
  PA_KV_NVFP4 = 2   /* pa_cache_write_nvfp4 / pa_decode_nvfp4 only */
} pa_kv_dtype;

/* Bits of the per-device error word (pa_get_device_error). */
#define PA_DEVERR_BAD_BLOCK_ID 0x1u /* table entry outside [0, num_blocks)  */
#define PA_DEVERR_BAD_SEQ_LEN  0x2u /* seq_len < 0 or > table capacity      */
#define PA_DEVERR_BAD_SLOT     0x4u /* slot >= num_blocks * block_size      */
#define PA_DEVERR_BAD_PAIR     0x8u /* copy pair id/length outside the pool */
#define PA_DEVERR_TIMEOUT      0x10u /* a pipeline wait hit its bound       */
#define PA_DEVERR_LAUNCH       0x20u /* internal launch-layout check failed */

/* Version of this ABI; bumped on any incompatible change. */
int32_t pa_abi_version(void);

/* Static, human-readable name of a status code. */
const char* pa_status_string(pa_status status);

/* Read and clear the current device's error word (bits PA_DEVERR_*).
 * Synchronises the current device.  `err` (host) receives the bits. */
pa_status pa_get_device_error(uint32_t* err);

/* ------------------------------------------------------------------ cache
 * pa_cache_write -- scatter this step's new K/V into the cache.
 * "Paged Attention and KV Cache Fragmentation", section "How PagedAttention
 * maps an OS concept onto GPU memory": new tokens land in the block the
 * table names for their position.  For each token t < num_tokens with
 * s = slot_mapping[t] >= 0:
 *     k_cache[s / block_size][h][s % block_size][:] = k_new[t][h][:]
 *     v_cache[s / block_size][h][s % block_size][:] = v_new[t][h][:]
 * for every KV head h, copied bit for bit.  Negative slots are skipped.
 *   k_new, v_new   device bf16 [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping   device int64 [num_tokens]
 *   k_cache/v_cache device bf16 pools (layout above)
 * Slots >= num_blocks * block_size are skipped and flag
 * PA_DEVERR_BAD_SLOT.  Two tokens naming the same slot give an unspecified
 * winner.  kv_dtype must be PA_KV_BF16 (FP8 caches: pa_cache_write_fp8,
 * else PA_ERR_UNSUPPORTED).
 * head_dim must be a multiple of 8. */
pa_status pa_cache_write(const void* k_new, const void* v_new,
                         const int64_t* slot_mapping, int32_t num_tokens,
                         void* k_cache, void* v_cache, int32_t num_blocks,
                         int32_t num_kv_heads, int32_t block_size,
                         int32_t head_dim, pa_kv_dtype kv_dtype, void* stream);

/* pa_cache_write_fp8 -- append this step's new K/V to an FP8 E4M3 cache.
 * "Paged Attention and KV Cache Fragmentation", section "Quantization as
 * a way to stretch paged memory further" (FP8 KV, fp32 scales); appending
 * into a partly filled block is this library's reading.  For each token t
 * with s = slot_mapping[t] >= 0, block = s / block_size, offset =
 * s % block_size, every KV head h, separately for K and V, with
 * s_t = max|x| / 448 over the token's row x (fp32):
 *   offset 0:          scale = s_t (1 if x is all zero)
 *   s_t > scale:       scale = s_t; rows r < offset are requantised,
 *                      code = e4m3(fp32(decode(code) * old) / scale)
 *   otherwise:         the scale is kept
 *   row offset:        code = e4m3(x / scale)
 * (fp32 IEEE multiply and divide, E4M3 round-to-nearest-even, saturating
 * to +-448.)  Filling a block in falling-absmax order reproduces
 * pa_quantize_fp8 exactly; in any order the final scale is the block's.
 *   k_new, v_new   device bf16 [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping   device int64 [num_tokens]
 *   k_cache/v_cache device uint8 E4M3 pools [num_blocks][Hkv][bs][head_dim]
 *   k_scale/v_scale device float [num_blocks][num_kv_heads], updated
 * The tokens of one call must name distinct blocks; slots >= num_blocks *
 * block_size are skipped and flag PA_DEVERR_BAD_SLOT.  head_dim in
 * {64, 128}. */
pa_status pa_cache_write_fp8(const void* k_new, const void* v_new,
                             const int64_t* slot_mapping, int32_t num_tokens,
                             void* k_cache, void* v_cache, float* k_scale,
                             float* v_scale, int32_t num_blocks,
                             int32_t num_kv_heads, int32_t block_size,
                             int32_t head_dim, void* stream);

/* pa_swap_out / pa_swap_in -- move whole cache blocks to host memory and
 * back.  "Paged Attention and KV Cache Fragmentation", section
 * "Offloading paged KV blocks to CPU DRAM and NVMe": blocks can move down
 * to host memory for headroom and come back when needed.  For i < num_ids and
 * b = block_ids[i]:
 *   swap_out: host_k[i] = k_cache[b], host_v[i] = v_cache[b] (all heads,
 *             slots and columns), and for FP8 caches host_k_scale[i][h] =
 *             k_scale[b][h] (likewise v);
 *   swap_in:  the reverse, into block b.
 * The host buffers ([num_ids][num_kv_heads][block_size][head_dim] of the
 * cache's element type, and [num_ids][num_kv_heads] floats) must be pinned
 * (cudaHostAlloc / cudaHostRegister) or managed: the kernel reads or
 * writes them in place, over NVLink-C2C on a Grace host, with no per-block
 * copy calls.  block_ids is device int32; ids outside the pool are skipped
 * and flag PA_DEVERR_BAD_BLOCK_ID.  Caches and host buffers 16-byte
 * aligned; head_dim * element size a multiple of 16.  Asynchronous on
 * `stream`; the host data is complete when the stream has reached it. */
pa_status pa_swap_out(const void* k_cache, const void* v_cache,
                      const float* k_scale, const float* v_scale,
                      const int32_t* block_ids, int32_t num_ids, void* host_k,
                      void* host_v, float* host_k_scale, float* host_v_scale,
                      int32_t num_blocks, int32_t num_kv_heads,
                      int32_t block_size, int32_t head_dim,
                      pa_kv_dtype kv_dtype, void* stream);
pa_status pa_swap_in(const void* host_k, const void* host_v,
                     const float* host_k_scale, const float* host_v_scale,
                     const int32_t* block_ids, int32_t num_ids, void* k_cache,
                     void* v_cache, float* k_scale, float* v_scale,
                     int32_t num_blocks, int32_t num_kv_heads, int32_t block_size,
                     int32_t head_dim, pa_kv_dtype kv_dtype, void* stream);

/* pa_copy_blocks -- copy-on-write of shared partial blocks.
 * "Paged Attention and KV Cache Fragmentation", section "How PagedAttention
 * maps an OS concept onto GPU memory": sequences sharing physical blocks
 * diverge only where their content differs.  For each pair p:
 *     (src, dst, n) = pairs[3p], pairs[3p+1], pairs[3p+2]
 *     cache[dst][h][0:n][:] = cache[src][h][0:n][:]  for all heads, K and V
 * and, for FP8 caches, k_scale[dst][h] = k_scale[src][h] (likewise v).
 *   pairs          device int32 [num_pairs][3] (pa_seq_append_slots output)
 *   k_scale/v_scale device float pools or NULL (must be non-NULL for FP8)
 * Pairs with an id outside the pool or n outside [0, block_size] are
 * skipped and flag PA_DEVERR_BAD_PAIR.  Pairs must not overlap (no dst may
 * be another pair's src). */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, float* k_scale,
                         float* v_scale, const int32_t* pairs,
                         int32_t num_pairs, int32_t num_blocks,
                         int32_t num_kv_heads, int32_t block_size,
                         int32_t head_dim, pa_kv_dtype kv_dtype, void* stream);

/* pa_quantize_fp8 -- build FP8 E4M3 cache blocks from bf16 blocks.
 * "Paged Attention and KV Cache Fragmentation", section "Quantization as a
 * way to stretch paged memory further" (FP8 halves the KV footprint).  For
 * each listed block b = block_ids[i] with n = valid_lens[i] valid tokens,
 * each KV head h, separately for K and V:
 *     a     = max |x| over tokens [0, n) and the head dimension (fp32)
 *     scale = a / 448 (IEEE fp32 division), or 1 when a == 0
 *     dst[b][h][t][:] = e4m3_rne_satfinite(src[b][h][t][:] / scale), t < n
 *     dst[b][h][t][:] = 0 (code +0), n <= t < block_size
 *     scale_out[b][h] = scale
 *   k_src, v_src    device bf16 pools; k_dst, v_dst device uint8 pools
 *   block_ids, valid_lens device int32 [num_ids]
 * Ids outside the pool or n outside [0, block_size] are skipped and flag
 * PA_DEVERR_BAD_BLOCK_ID. */
pa_status pa_quantize_fp8(const void* k_src, const void* v_src,
                          const int32_t* block_ids, const int32_t* valid_lens,
                          int32_t num_ids, uint8_t* k_dst, uint8_t* v_dst,
                          float* k_scale, float* v_scale, int32_t num_blocks,
                          int32_t num_kv_heads, int32_t block_size,
                          int32_t head_dim, void* stream);

/* ----------------------------------------------------------------- decode
 * pa_decode_workspace_size -- bytes of device workspace pa_decode needs for
 * this shape with `num_splits` work partitions (0 = the automatic choice
 * for the current device, the largest over the cache formats: the same
 * size serves pa_decode, pa_decode_append(_fp8), pa_decode_nvfp4).  Writes
 * the size to *bytes (host). */
pa_status pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim,
                                   int32_t num_splits, size_t* bytes);

/* pa_decode -- single-token paged decode attention.
 * "KV cache fragmentation" (field guide), section "Definition" (the kernel
 * walks the page table) and "Paged Attention and KV Cache Fragmentation",
 * section "How PagedAttention maps an OS concept onto GPU memory" (a request
 * sees its cache as one continuous sequence).  For every sequence b and
 * query head h, with g = h / (num_q_heads / num_kv_heads) and
 * n = seq_lens[b]:
 *     K_b[t] = k_cache[block_tables[b][t / block_size]][g][t % block_size]
 *     s_t    = scale * <q[b][h], K_b[t]>,           0 <= t < n
 *     out[b][h] = sum_t softmax(s)_t * V_b[t]       (bf16 result)
 * with fp32 accumulation throughout.  FP8 caches dequantise as
 * decode(code) * k_scale[block][g] (likewise V); the query and the softmax
 * weights meet the E4M3 codes on the tensor cores as two-term E4M3 splits
 * (hi + lo / 16 after a power-of-two row scale: exact for a bf16 query
 * except below about 2^-14 of its row's largest element; each softmax
 * weight within 2^-8 of itself plus 2^-18 of the largest), with fp32
 * products and sums.  A sequence with n == 0
 * yields zeros.  Long contexts are split over up to `num_splits` persistent
 * work partitions (0 = automatic) whose partial results are merged with a
 * log-sum-exp reduction; the split points depend only on seq_lens, so the
 * result does not depend on which physical blocks the tables name.
 *   q            device bf16 [num_seqs][num_q_heads][head_dim]
 *   k_cache, v_cache device pools of kv_dtype; num_blocks = pool blocks
 *   k_scale, v_scale device float [num_blocks][num_kv_heads] (FP8) or NULL
 *   block_tables device int32 [num_seqs][max_blocks_per_seq]
 *   seq_lens     device int32 [num_seqs]
 *   out          device bf16 [num_seqs][num_q_heads][head_dim]
 *   workspace    device buffer of >= pa_decode_workspace_size() bytes
 *                (contents need no initialisation; may be NULL if the size
 *                is 0)
 * Supported: head_dim in {64, 128}; 1 <= num_q_heads / num_kv_heads <= 8;
 * block_size a power of two in [8, 256].  Table entries outside the pool
 * read as zeros and flag PA_DEVERR_BAD_BLOCK_ID; seq_lens outside
 * [0, max_blocks_per_seq * block_size] are clamped and flag
 * PA_DEVERR_BAD_SEQ_LEN. */
pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                    const float* k_scale, const float* v_scale,
                    pa_kv_dtype kv_dtype, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* seq_lens,
                    int32_t num_seqs, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim,
                    int32_t block_size, int32_t num_blocks, float scale,
                    void* out, void* workspace, size_t workspace_bytes,
                    int32_t num_splits, void* stream);

/* pa_decode_append -- this step's cache write and decode in one launch.
 * The same result, in the cache and in out, as
 *     pa_cache_write(k_new, v_new, slot_mapping, num_seqs, ...);
 *     pa_decode(q, k_cache, v_cache, ..., PA_KV_BF16, ...);
 * for a decode step where sequence b appends one token (row b of
 * k_new/v_new) at its last position: "Paged Attention and KV Cache
 * Fragmentation", section "How PagedAttention maps an OS concept onto GPU
 * memory" (a new token lands in the block the table names for its
 * position, then the kernel walks the table).  The CTA that owns sequence
 * b's last tile stores the row just before it copies that tile.
 *   k_new, v_new   device bf16 [num_seqs][num_kv_heads][head_dim]
 *   slot_mapping   device int64 [num_seqs]; < 0: sequence b appends nothing
 *   other arguments as pa_decode, with a bf16 cache (no scales)
 * Requirements, beyond pa_decode's: slot_mapping[b] >= 0 must be the slot
 * of position seq_lens[b] - 1 (block_tables[b][(n-1)/bs] * bs + (n-1) % bs,
 * as the block manager returns it), and that block must be private to b
 * (copy-on-write done).  A slot elsewhere, or on an empty sequence, is not
 * written and flags PA_DEVERR_BAD_SLOT.  FP8 caches: pa_decode_append_fp8. */
pa_status pa_decode_append(const void* q, const void* k_new, const void* v_new,
                           const int64_t* slot_mapping, void* k_cache,
                           void* v_cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* seq_lens,
                           int32_t num_seqs, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks, float scale,
                           void* out, void* workspace, size_t workspace_bytes,
                           int32_t num_splits, void* stream);

/* pa_decode_append_fp8 -- pa_decode_append for an FP8 E4M3 cache: the same
 * cache (codes and scales) and output as
 *     pa_cache_write_fp8(k_new, v_new, slot_mapping, num_seqs, ...);
 *     pa_decode(q, k_cache, v_cache, k_scale, v_scale, PA_KV_FP8_E4M3, ...);
 * bit for bit.  head_dim 64: the CTA that copies sequence b's last tile
 * first quantises the new row into its block (growing the block's scale
 * and requantising its earlier rows when needed), which is exact only when
 * that tile holds the whole block.  head_dim 128: two launches on `stream`,
 * the FP8 cache write (with the slot check below) and then pa_decode's
 * tensor-core kernel.  block_size must be 8 or 16 (else
 * PA_ERR_UNSUPPORTED).  k_scale / v_scale are read and updated.  Other
 * arguments and requirements as pa_decode_append, including its slot check:
 * a slot that is not the one of position seq_lens[b] - 1 is not written and
 * flags PA_DEVERR_BAD_SLOT. */
pa_status pa_decode_append_fp8(const void* q, const void* k_new, const void* v_new,
                               const int64_t* slot_mapping, void* k_cache,
                               void* v_cache, float* k_scale, float* v_scale,
                               const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* seq_lens,
                               int32_t num_seqs, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int32_t num_blocks, float scale,
                               void* out, void* workspace, size_t workspace_bytes,
                               int32_t num_splits, void* stream);

/* --------------------------------------------------------------- NVFP4
 * NVFP4 caches.  "Paged Attention and KV Cache Fragmentation", section
 * "Quantization as a way to stretch paged memory further", names NVFP4 as
 * the Blackwell cache format that halves FP8's footprint again, without
 * defining it.  This library takes NVIDIA's published NVFP4: FP4 E2M1
 * values (0, 0.5, 1, 1.5, 2, 3, 4, 6 and negatives), one E4M3 scale per 16
 * consecutive values of a head row, and one fp32 scale S per tensor (the K,
 * resp. V, cache of a layer) that the caller calibrates, e.g. S = amax /
 * (6 * 448).  A row x (bf16, widened to fp32) is stored as
 *     s_g = e4m3(max|x_g| / (6 S))   for each 16-value group g
 *     q_i = e2m1(x_i / (e4m3(s_g) * S))   (0 when s_g decodes to 0)
 * (fp32 IEEE multiply and divide; both encoders round to nearest even and
 * saturate, E4M3 to 448, E2M1 to 6) and reads back as
 * e2m1(q_i) * e4m3(s_g) * S.  Layout per (block, KV head), bs = block_size,
 * D = head_dim, all uint8:
 *     k_cache [num_blocks][Hkv][bs][D/2]    byte j of token t holds values
 *                                           2j (low nibble) and 2j+1
 *     k_sf    [num_blocks][Hkv][bs][D/16]   E4M3 scale of group g of token t
 *     v_cache [num_blocks][Hkv][bs/2][D]    byte d of pair-row p holds token
 *                                           2p (low nibble) and 2p+1 of
 *                                           dimension d
 *     v_sf    [num_blocks][Hkv][D/16][bs]   E4M3 scale of group g of token t
 * 4.5 bits per value.  Supported: head_dim in {64, 128}; block_size a power
 * of two in [16, 256]; 1 <= num_q_heads / num_kv_heads <= 8.
 *
 * pa_cache_write_nvfp4 -- quantise and store this step's new K/V.  For each
 * token t < num_tokens with s = slot_mapping[t] >= 0, every KV head h: the
 * K row k_new[t][h] and the V row v_new[t][h] are quantised as above into
 * block s / bs, token s % bs.  Slots must be distinct; slots >= num_blocks
 * * block_size are skipped and flag PA_DEVERR_BAD_SLOT.
 *   k_new, v_new         device bf16 [num_tokens][num_kv_heads][head_dim]
 *   slot_mapping         device int64 [num_tokens]
 *   k_cache..v_sf        device pools (layout above), updated in place
 *   k_gscale, v_gscale   the tensor scales S (host floats, > 0, finite) */
pa_status pa_cache_write_nvfp4(const void* k_new, const void* v_new,
                               const int64_t* slot_mapping, int32_t num_tokens,
                               void* k_cache, void* v_cache, void* k_sf, void* v_sf,
                               float k_gscale, float v_gscale, int32_t num_blocks,
                               int32_t num_kv_heads, int32_t block_size,
                               int32_t head_dim, void* stream);

/* pa_decode_nvfp4 -- pa_decode over an NVFP4 cache: the same attention,
 * with K_b[t] and V_b[t] the dequantised rows e2m1 * e4m3 block scale * S.
 * Accumulation in fp32; K and V reach the tensor cores as f16 values, which
 * hold every e2m1 * e4m3 product exactly; q is rounded to f16 (|q| must
 * stay below 65504).  The workspace is pa_decode_workspace_size()'s.
 * Other arguments, results and device-error behaviour as pa_decode. */
pa_status pa_decode_nvfp4(const void* q, const void* k_cache, const void* v_cache,
                          const void* k_sf, const void* v_sf, float k_gscale,
                          float v_gscale, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, const int32_t* seq_lens,
                          int32_t num_seqs, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int32_t num_blocks, float scale,
                          void* out, void* workspace, size_t workspace_bytes,
                          int32_t num_splits, void* stream);

/* pa_decode_append_nvfp4 -- the NVFP4 decode step in one launch: the same
 * pools and output, bit for bit, as
 *     pa_cache_write_nvfp4(k_new, v_new, slot_mapping, num_seqs, ...);
 *     pa_decode_nvfp4(q, k_cache, v_cache, k_sf, v_sf, ...);
 * where row b of k_new / v_new ([num_seqs][num_kv_heads][head_dim] bf16) is
 * sequence b's new token.  The CTA that copies a (sequence, KV head)'s last
 * tile first quantises that head's new rows into it.  Requirements as
 * pa_decode_append: slot_mapping[b] >= 0 must be the slot of position
 * seq_lens[b] - 1 in a block private to b; another slot, or one on an empty
 * sequence, is not written and flags PA_DEVERR_BAD_SLOT; < 0 appends nothing.
 * The pools are read and written; other arguments as pa_decode_nvfp4. */
pa_status pa_decode_append_nvfp4(const void* q, const void* k_new, const void* v_new,
                                 const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                 void* k_sf, void* v_sf, float k_gscale, float v_gscale,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* seq_lens, int32_t num_seqs,
                                 int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                 float scale, void* out, void* workspace,
                                 size_t workspace_bytes, int32_t num_splits, void* stream);

/* pa_decode_cascade -- pa_decode for a batch whose sequences all start with
 * the same prefix_len tokens in the same physical blocks (forks of one
 * prompt): "Paged Attention and KV Cache Fragmentation", section "How
 * PagedAttention maps an OS concept onto GPU memory", and the "KV cache
 * fragmentation" field guide, section "Why it matters" (sequences sharing
 * a prefix point at the same blocks).  The result equals pa_decode's
 * (bf16 cache): softmax attention over every token of each sequence.  The
 * prefix is read once for all sequences -- its attention partial for every
 * (sequence, query head) is a dense product of all query rows with the
 * prefix keys and values on the tensor cores -- and each sequence's tokens
 * past the prefix run through the paged decode, which folds the prefix
 * partial in by a log-sum-exp merge.
 *   prefix_len   a multiple of 16 and of block_size, <= the table width; the
 *                prefix blocks are read from block_tables[0] and must be
 *                the first prefix_len / block_size entries of every row
 *   seq_lens[b]  >= prefix_len (shorter ones give zeros and flag
 *                PA_DEVERR_BAD_SEQ_LEN)
 *   workspace    >= pa_decode_cascade_workspace_size() bytes (same
 *                shapes, block_size, prefix_len and num_splits), 16-byte
 *                aligned (no initialisation needed)
 * other arguments as pa_decode.  prefix_len == 0 is plain pa_decode. */
pa_status pa_decode_cascade_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_dim,
                                           int32_t block_size, int32_t prefix_len,
                                           int32_t num_splits, size_t* bytes);
pa_status pa_decode_cascade(const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens,
                            int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks,
                            int32_t prefix_len, float scale, void* out,
                            void* workspace, size_t workspace_bytes,
                            int32_t num_splits, void* stream);

/* pa_decode_noalloc -- pa_decode for callers that cannot allocate.
 * The pages have no counterpart: this is a library-only convenience.
 * Some callers cannot call cudaMalloc or otherwise obtain device memory:
 * plugin hosts that forbid allocation inside their execute callback and
 * provide no workspace, services that fix their whole device-memory budget
 * at start-up, and thin foreign-function callers with no device allocator.
 * This entry point takes the same arguments as pa_decode minus the
 * workspace pointer and size, and uses instead a
 * library-owned device array of PA_NOALLOC_SCRATCH_BYTES (16 MiB) that every
 * GPU which loads the library holds until the process exits.
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library
 *     routine is called.
 *   - The first call on each device looks up that device's address of the
 *     array (with the device current); make that first call before any
 *     stream capture on the device.
 *   - The limit applies to the workspace this call itself needs: that of
 *     its own KV format at its partition count (num_splits, or with 0 the
 *     format's automatic count, one partition per resident decode CTA).  A
 *     call needing more than PA_NOALLOC_SCRATCH_BYTES is rejected with
 *     PA_ERR_WORKSPACE and nothing is enqueued.  pa_decode_workspace_size
 *     with num_splits = 0 returns the largest automatic size over all
 *     formats, so as a pre-check it can only over-predict a refusal.
 *   - All calls on a device share the one array, which keeps whatever the
 *     last call left in it.  Nothing in it needs to start at zero: every
 *     partial result a call reads was written earlier by the same call.
 *   - Calls whose kernels overlap on the GPU (different streams without
 *     ordering between them) race on the array; order them on one stream
 *     or use pa_decode with separate workspaces. */
#define PA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
pa_status pa_decode_noalloc(const void* q, const void* k_cache,
                            const void* v_cache, const float* k_scale,
                            const float* v_scale, pa_kv_dtype kv_dtype,
                            const int32_t* block_tables,
                            int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, int32_t num_seqs,
                            int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size,
                            int32_t num_blocks, float scale, void* out,
                            int32_t num_splits, void* stream);

/* ------------------------------------------------------- block manager
 * Host-only block allocator ("Paged Attention and KV Cache Fragmentation",
 * section "How PagedAttention maps an OS concept onto GPU memory"; shared
 * prefixes and forks: "KV cache fragmentation", section "Why it matters").
 * A LIFO free list (a fresh allocator hands out 0, 1, 2, ...) and one
 * refcount per block.  Every call is all-or-nothing: on any error no state
 * changes.  No device memory is touched.  The handle is not thread-safe. */
typedef struct pa_allocator pa_allocator;

/* Create an allocator over blocks [0, num_blocks); *out receives it. */
pa_status pa_allocator_create(int32_t num_blocks, pa_allocator** out);
/* Destroy an allocator (NULL is a no-op). */
void pa_allocator_destroy(pa_allocator* a);
/* Pop n blocks (refcount 1 each) into ids_out[0..n); OUT_OF_BLOCKS if fewer
 * than n are free. */
pa_status pa_block_alloc(pa_allocator* a, int32_t n, int32_t* ids_out);
/* Drop one reference per listed id (ids may repeat); blocks reaching zero
 * are pushed on the free list in list order.  BAD_BLOCK_ID if an id is
 * outside the pool or listed more often than it is referenced. */
pa_status pa_block_free(pa_allocator* a, const int32_t* ids, int32_t n);
/* Add one reference per listed id (a forked sequence shares the blocks).
 * BAD_BLOCK_ID if an id is outside the pool or free. */
pa_status pa_block_fork(pa_allocator* a, const int32_t* ids, int32_t n);
/* Current refcount of one block. */
pa_status pa_block_refcount(const pa_allocator* a, int32_t id, int32_t* rc);
/* Number of free blocks (-1 for a NULL handle). */
int32_t pa_block_num_free(const pa_allocator* a);

/* pa_seq_append_slots -- grow one sequence from `len` to `len + n` tokens.
 * table (host int32 [max_blocks]) holds the sequence's block ids; entries
 * [0, ceil(len / block_size)) must be live.  If the last held block is
 * partially filled and shared (refcount > 1), it is first replaced by a
 * fresh block and one copy request (src, dst, len % block_size) is written
 * to cow_pair_out[0..3) with *num_cow = 1 (else *num_cow = 0); the caller
 * runs pa_copy_blocks on it before writing the new tokens.  Then a block is
 * allocated for every block boundary the new tokens cross, and
 * slots_out[i] = table[p / block_size] * block_size + p % block_size for
 * p = len + i.  INVALID_ARG if ceil((len + n) / block_size) > max_blocks;
 * OUT_OF_BLOCKS if the free list cannot cover the copy and the growth. */
pa_status pa_seq_append_slots(pa_allocator* a, int32_t* table,
                              int32_t max_blocks, int32_t len, int32_t n,
                              int32_t block_size, int64_t* slots_out,
                              int32_t* cow_pair_out, int32_t* num_cow);

/* pa_batch_append_slots -- one step's appends for a whole batch in one call:
 * for i = 0, 1, ..., num_seqs - 1 in order, sequence i (row i of tables,
 * host int32 [num_seqs][max_blocks]) grows from lens[i] by n_new[i] tokens
 * exactly as pa_seq_append_slots would.  slots_out (host int64,
 * sum(n_new) entries) receives the slots sequence after sequence;
 * cow_pairs_out (host int32 [num_seqs][3]) and n_cow_out[i] each
 * sequence's copy request.  The first sequence that fails stops the batch:
 * its status is returned, *num_done (host) = i, sequences >= i are
 * untouched and sequences < i keep their appends (each one is
 * all-or-nothing, the batch is not).  On success *num_done = num_seqs. */
pa_status pa_batch_append_slots(pa_allocator* a, int32_t* tables,
                                int32_t max_blocks, const int32_t* lens,
                                const int32_t* n_new, int32_t num_seqs,
                                int32_t block_size, int64_t* slots_out,
                                int32_t* cow_pairs_out, int32_t* n_cow_out,
                                int32_t* num_done);

/* pa_allocator_usage -- how full the reserved blocks are.  "KV cache
 * fragmentation" field guide, section "Why it matters", and "Paged
 * Attention and KV Cache Fragmentation", section "How PagedAttention maps
 * an OS concept onto GPU memory": a paged cache wastes at most each
 * sequence's unfilled last block, where a contiguous one reserves every
 * request's maximum length.  For the sequences given (host tables
 * [num_seqs][max_blocks], lengths lens[num_seqs]):
 *   out[0] live_blocks     blocks of the allocator with refcount > 0
 *   out[1] slots_reserved  live_blocks * block_size
 *   out[2] tokens_stored   distinct (block, offset) slots holding a token of
 *                          some sequence (shared blocks counted once)
 *   out[3] tokens_logical  sum of lens
 * BAD_BLOCK_ID if a table entry a length reaches is not live. */
pa_status pa_allocator_usage(const pa_allocator* a, const int32_t* tables,
                             int32_t max_blocks, const int32_t* lens,
                             int32_t num_seqs, int32_t block_size,
                             int64_t* out);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
