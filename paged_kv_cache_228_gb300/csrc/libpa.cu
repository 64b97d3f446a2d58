// libpa: C ABI entry points (declared in include/pa.h).  Host-side argument
// validation, TMA descriptor encoding and kernel launches; the kernels live
// in decode.cuh, nvfp4.cuh, cascade.cuh and cache_ops.cuh, the host block
// manager in
// block_manager.cpp.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "cache_ops.cuh"
#include "cascade.cuh"
#include "decode.cuh"
#include "decode_tc.cuh"
#include "nvfp4.cuh"
#include "pa.h"
#include "pa_testing.h"

namespace pa {

namespace {

constexpr int kMaxDevices = 64;

// An NVTX range named after the entry point around its host work and
// launches (a profiler shows it; without one it costs a no-op call).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline bool pow2_in(int32_t x, int32_t lo, int32_t hi) {
  return x >= lo && x <= hi && (x & (x - 1)) == 0;
}

inline int ilog2(int32_t x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

struct DeviceInfo {
  bool init = false;
  int sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

// Polls before a decode kernel's pipeline wait gives up, and the stall test
// hook (pa_testing_set_wait_limit).
constexpr uint32_t kDefaultWaitLimit = 1u << 22;
std::atomic<uint32_t> g_wait_limit{kDefaultWaitLimit};
std::atomic<int32_t> g_wait_stall{0};

pa_status device_sms(int* sms, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev[dev].init) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PA_ERR_CUDA;
    g_dev[dev].sms = n;
    g_dev[dev].init = true;
  }
  *sms = g_dev[dev].sms;
  if (dev_out) *dev_out = dev;
  return PA_OK;
}

// Launch as a programmatic dependent of the previous work in the stream:
// the grid may start launching before that work ends, and waits for it on
// the device (griddepcontrol.wait) before it reads anything.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 2D map over a row-major [rows][inner] array; box = [box_inner, box_rows].
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base,
               uint64_t inner, uint64_t rows, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Decode launch plan for one (head_dim, dtype) instantiation: as many CTAs
// of its shape per SM as registers allow up to kMaxCtasPerSm, each with the
// deepest stage ring that lets that many share the SM's shared memory.
constexpr int kMaxCtasPerSm = 16;
constexpr size_t kSmemPerSm = 228 * 1024;
constexpr size_t kSmemReservedPerCta = 1024;

using DecodeFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, DecodeParams);

template <int D, bool FP8>
DecodeFn decode_fn(bool append = false) {
  if (DecodeShape<D, FP8>::kTwoWarps) return paged_decode_ws_kernel<D, FP8>;
  return append ? paged_decode_kernel<D, FP8, true> : paged_decode_kernel<D, FP8, false>;
}

struct DecodePlan {
  int ctas_per_sm = 0;
  int stages = 0;
};

template <int D, bool FP8>
pa_status decode_plan(int dev, DecodePlan* out) {
  using L = Smem<D, FP8>;
  static DecodePlan cached[kMaxDevices];
  std::lock_guard<std::mutex> lk(g_mu);
  DecodePlan& pl = cached[dev];
  if (pl.ctas_per_sm == 0) {
    const DecodeFn fn = decode_fn<D, FP8>();
    const int threads = DecodeShape<D, FP8>::kThreads;
    // CTAs per SM that registers (and the thread/CTA limits) allow
    int by_regs = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&by_regs, fn, threads, 0) != cudaSuccess)
      return PA_ERR_CUDA;
    const int want = by_regs < kMaxCtasPerSm ? by_regs : kMaxCtasPerSm;
    if (want < 1) return PA_ERR_UNSUPPORTED;
    const size_t per_cta = kSmemPerSm / want - kSmemReservedPerCta;
    int s = static_cast<int>((per_cta - decode_smem_bytes<D, FP8>(0)) / L::kStageBytes);
    if (s < 2) s = 2;
    if (s > kMaxStages) s = kMaxStages;
    const size_t smem = decode_smem_bytes<D, FP8>(s);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return PA_ERR_CUDA;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess)
      return PA_ERR_CUDA;
    if (n < 1) return PA_ERR_UNSUPPORTED;
    pl.stages = s;
    pl.ctas_per_sm = n;
  }
  *out = pl;
  return PA_OK;
}

// The tcgen05 FP8 decode: kTcCtasPerSm CTAs per SM (if registers allow),
// each with the deepest ring of 32 KB chunk stages that lets them share the
// SM's shared memory.
constexpr int kTcCtasPerSm = 1;

template <int D>
pa_status tc_plan(int dev, DecodePlan* out) {
  static DecodePlan cached[kMaxDevices];
  std::lock_guard<std::mutex> lk(g_mu);
  DecodePlan& pl = cached[dev];
  if (pl.ctas_per_sm == 0) {
    const size_t per_cta = kSmemPerSm / kTcCtasPerSm - kSmemReservedPerCta;
    int s = static_cast<int>((per_cta - tc_smem_bytes<D>(0)) / TcSmem<D>::kStage);
    if (s < 2) s = 2;
    if (s > kTcMaxStages) s = kTcMaxStages;
    const size_t smem = tc_smem_bytes<D>(s);
    if (cudaFuncSetAttribute(paged_decode_tc_fp8_kernel<D>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return PA_ERR_CUDA;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_decode_tc_fp8_kernel<D>,
                                                      kTcThreads, smem) != cudaSuccess)
      return PA_ERR_CUDA;
    if (n < 1) return PA_ERR_UNSUPPORTED;
    pl.stages = s;
    pl.ctas_per_sm = n < kTcCtasPerSm ? n : kTcCtasPerSm;
  }
  *out = pl;
  return PA_OK;
}

// NVFP4 decode: a fixed ring depth per head_dim, so the plan is the CTAs
// per SM that registers and that ring allow (at most kMaxCtasPerSm).
template <int D>
pa_status fp4_plan(int dev, int* ctas_per_sm) {
  static int cached[kMaxDevices] = {0};
  std::lock_guard<std::mutex> lk(g_mu);
  if (cached[dev] == 0) {
    const size_t smem = fp4_smem_bytes<D>();
    if (cudaFuncSetAttribute(paged_decode_nvfp4_kernel<D, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(paged_decode_nvfp4_kernel<D, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return PA_ERR_CUDA;
    // the plain instantiation sets the grid; the append one launches the same
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_decode_nvfp4_kernel<D, false>,
                                                      32, smem) != cudaSuccess)
      return PA_ERR_CUDA;
    if (n < 1) return PA_ERR_UNSUPPORTED;
    cached[dev] = n < kMaxCtasPerSm ? n : kMaxCtasPerSm;
  }
  *ctas_per_sm = cached[dev];
  return PA_OK;
}

// What the work split charges per (sequence, KV head) segment, in units
// of kUnit = 8 per work unit: the segment's query copy, first table batch
// and finish.  Two tiles' worth was the best of 8..24 on every kernel shape
// on the Llama-3.1-8B-shaped layer (~837 tokens a sequence).  The tcgen05
// FP8 kernel's work unit is a 256-token chunk; per-CTA timestamps on that
// layer fit 1.0 us per chunk and 0.7 us per piece of a segment.
constexpr int32_t kSegCostBf16 = 16;
constexpr int32_t kSegCostFp8 = 16;
constexpr int32_t kSegCostFp4 = 16;
constexpr int32_t kSegCostTc = 6;

// Workspace for P decode CTAs over `segs` segments: P + segs partial
// slots (a CTA's pieces never collide: piece = cta + segment), then P
// merge jobs.
size_t workspace_bytes_for(int64_t P, int64_t segs, int32_t head_dim) {
  const int64_t pieces = P + segs;
  return static_cast<size_t>(pieces) * kMaxG *
             (static_cast<size_t>(head_dim) * sizeof(float) + sizeof(float2)) +
         static_cast<size_t>(P) * sizeof(int2);
}

template <int D, bool FP8>
pa_status launch_decode(const DecodeParams& prm_in, const void* q,
                        const void* k_cache, const void* v_cache,
                        void* workspace, size_t workspace_bytes,
                        int32_t num_splits, cudaStream_t stream) {
  int sms = 0, dev = 0;
  pa_status st = device_sms(&sms, &dev);
  if (st != PA_OK) return st;
  DecodePlan plan;
  st = decode_plan<D, FP8>(dev, &plan);
  if (st != PA_OK) return st;
  const int stages = plan.stages;
  const int32_t P = num_splits > 0 ? num_splits : sms * plan.ctas_per_sm;
  const int64_t segs = static_cast<int64_t>(prm_in.num_seqs) * prm_in.num_kv_heads;
  const size_t need = P > 1 ? workspace_bytes_for(P, segs, D) : 0;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
    return PA_ERR_WORKSPACE;

  DecodeParams prm = prm_in;
  prm.num_ctas = P;
  prm.seg_cost = FP8 ? kSegCostFp8 : kSegCostBf16;
  prm.stages = stages;
  prm.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  prm.stall = g_wait_stall.load(std::memory_order_relaxed);
  prm.ws_o = nullptr;
  prm.ws_ml = nullptr;
  prm.ws_job = nullptr;
  if (need > 0) {
    const int64_t pieces = P + segs;
    char* w = static_cast<char*>(workspace);
    prm.ws_o = reinterpret_cast<float*>(w);
    w += static_cast<size_t>(pieces) * kMaxG * D * sizeof(float);
    prm.ws_ml = reinterpret_cast<float2*>(w);
    w += static_cast<size_t>(pieces) * kMaxG * sizeof(float2);
    prm.ws_job = reinterpret_cast<int2*>(w);
  }

  CUtensorMap tq, tk, tv;
  const uint64_t qrows = static_cast<uint64_t>(prm.num_seqs) * prm.num_q_heads;
  if (!encode_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, D, qrows, D * 2, 64, 8,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return PA_ERR_CUDA;
  const uint32_t box_rows = prm.block_size < kTile ? prm.block_size : kTile;
  const uint64_t rows = static_cast<uint64_t>(prm.rows_total);
  if (FP8) {
    const CUtensorMapSwizzle sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!encode_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, k_cache, D, rows, D, D, box_rows, sw) ||
        !encode_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, v_cache, D, rows, D, D, box_rows, sw))
      return PA_ERR_CUDA;
  } else {
    if (!encode_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k_cache, D, rows, D * 2, 64, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v_cache, D, rows, D * 2, 64, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return PA_ERR_CUDA;
  }
  // Both grids are programmatic dependents of the work before them in the
  // stream, which hides the launch gaps.
  const bool append = prm.k_new != nullptr;
  if (append && !DecodeShape<D, FP8>::kTwoWarps) {
    // the append instantiation shares the plan's shared-memory size
    static bool attr_set[kMaxDevices] = {false};
    std::lock_guard<std::mutex> lk(g_mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(decode_fn<D, FP8>(true),
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(decode_smem_bytes<D, FP8>(stages))) != cudaSuccess)
        return PA_ERR_CUDA;
      attr_set[dev] = true;
    }
  }
  if (launch_pdl(decode_fn<D, FP8>(append), dim3(static_cast<unsigned>(P)),
                 dim3(DecodeShape<D, FP8>::kThreads), decode_smem_bytes<D, FP8>(stages), stream,
                 tq, tk, tv, prm) != cudaSuccess)
    return PA_ERR_CUDA;
  if (launch_pdl(paged_decode_merge_kernel<D>, dim3(static_cast<unsigned>(P)),
                 dim3(prm.group * D / 4), 0, stream, prm) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

// FP8 cache, head_dim 128, plain decode: the tcgen05 kernel and the merge.
template <int D>
pa_status launch_decode_tc(const DecodeParams& prm_in, const void* q, const void* k_cache,
                           const void* v_cache, void* workspace, size_t workspace_bytes,
                           int32_t num_splits, cudaStream_t stream) {
  int sms = 0, dev = 0;
  pa_status st = device_sms(&sms, &dev);
  if (st != PA_OK) return st;
  DecodePlan plan;
  st = tc_plan<D>(dev, &plan);
  if (st != PA_OK) return st;
  const int32_t P = num_splits > 0 ? num_splits : sms * plan.ctas_per_sm;
  const int64_t segs = static_cast<int64_t>(prm_in.num_seqs) * prm_in.num_kv_heads;
  const size_t need = P > 1 ? workspace_bytes_for(P, segs, D) : 0;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
    return PA_ERR_WORKSPACE;
  DecodeParams prm = prm_in;
  prm.num_ctas = P;
  prm.seg_cost = kSegCostTc;
  prm.tile_log2 = 4;  // the split in whole 256-token chunks
  prm.stages = plan.stages;
  prm.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  prm.stall = g_wait_stall.load(std::memory_order_relaxed);
  prm.ws_o = nullptr;
  prm.ws_ml = nullptr;
  prm.ws_job = nullptr;
  if (need > 0) {
    const int64_t pieces = P + segs;
    char* w = static_cast<char*>(workspace);
    prm.ws_o = reinterpret_cast<float*>(w);
    w += static_cast<size_t>(pieces) * kMaxG * D * sizeof(float);
    prm.ws_ml = reinterpret_cast<float2*>(w);
    w += static_cast<size_t>(pieces) * kMaxG * sizeof(float2);
    prm.ws_job = reinterpret_cast<int2*>(w);
  }
  CUtensorMap tq, tk, tv;
  const uint64_t qrows = static_cast<uint64_t>(prm.num_seqs) * prm.num_q_heads;
  const uint32_t box_rows = prm.block_size < kTile ? prm.block_size : kTile;
  const uint64_t rows = static_cast<uint64_t>(prm.rows_total);
  if (!encode_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, D, qrows, D * 2, 64, 8,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, k_cache, D, rows, D, D, box_rows,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, v_cache, D, rows, D, D, box_rows,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return PA_ERR_CUDA;
  if (launch_pdl(paged_decode_tc_fp8_kernel<D>, dim3(static_cast<unsigned>(P)),
                 dim3(kTcThreads), tc_smem_bytes<D>(plan.stages), stream, tq, tk, tv,
                 prm) != cudaSuccess)
    return PA_ERR_CUDA;
  if (launch_pdl(paged_decode_merge_kernel<D>, dim3(static_cast<unsigned>(P)),
                 dim3(prm.group * D / 4), 0, stream, prm) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int32_t pa_abi_version(void) { return 1; }

extern "C" pa_status pa_testing_set_wait_limit(uint32_t polls, int32_t stall) {
  if (polls == 0) {
    pa::g_wait_limit.store(pa::kDefaultWaitLimit);
    pa::g_wait_stall.store(0);
    return PA_OK;
  }
  if (stall != 0 && stall != 1) return PA_ERR_INVALID_ARG;
  pa::g_wait_limit.store(polls);
  pa::g_wait_stall.store(stall);
  return PA_OK;
}

extern "C" const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_OUT_OF_BLOCKS: return "PA_ERR_OUT_OF_BLOCKS";
    case PA_ERR_BAD_BLOCK_ID: return "PA_ERR_BAD_BLOCK_ID";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
  }
  return "PA_ERR_UNKNOWN";
}

extern "C" pa_status pa_get_device_error(uint32_t* err) {
  if (err == nullptr) return PA_ERR_INVALID_ARG;
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return PA_ERR_CUDA;
  *err = v;
  return PA_OK;
}

extern "C" pa_status pa_cache_write(const void* k_new, const void* v_new,
                                    const int64_t* slot_mapping, int32_t num_tokens,
                                    void* k_cache, void* v_cache, int32_t num_blocks,
                                    int32_t num_kv_heads, int32_t block_size,
                                    int32_t head_dim, pa_kv_dtype kv_dtype, void* stream) {
  const NvtxRange nvtx_range("pa_cache_write");
  if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0 || block_size <= 0 ||
      head_dim <= 0 || head_dim % 8 != 0)
    return PA_ERR_INVALID_ARG;
  if (kv_dtype == PA_KV_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  if (kv_dtype != PA_KV_BF16) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PA_ERR_INVALID_ARG;
  int sms = 0;
  pa_status st = device_sms(&sms, nullptr);
  if (st != PA_OK) return st;
  const int32_t cpr = head_dim / 8;
  const int64_t total = 2LL * num_tokens * num_kv_heads * cpr;
  int64_t grid = (total + 255) / 256;
  if (grid > static_cast<int64_t>(sms) * 16) grid = static_cast<int64_t>(sms) * 16;
  const cudaError_t e = launch_pdl(
      cache_write_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
      static_cast<cudaStream_t>(stream), static_cast<const uint4*>(k_new),
      static_cast<const uint4*>(v_new), slot_mapping, num_tokens, static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), static_cast<int64_t>(num_blocks) * block_size,
      num_kv_heads, block_size, cpr);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_cache_write_fp8(const void* k_new, const void* v_new,
                                        const int64_t* slot_mapping, int32_t num_tokens,
                                        void* k_cache, void* v_cache, float* k_scale,
                                        float* v_scale, int32_t num_blocks,
                                        int32_t num_kv_heads, int32_t block_size,
                                        int32_t head_dim, void* stream) {
  const NvtxRange nvtx_range("pa_cache_write_fp8");
  if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0 || block_size <= 0)
    return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_new) & 3u) || (reinterpret_cast<uintptr_t>(v_new) & 3u) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return PA_ERR_INVALID_ARG;
  const int64_t warps = 2LL * num_tokens * num_kv_heads;
  const int64_t grid = (warps * 32 + 255) / 256;
  if (grid > INT_MAX) return PA_ERR_UNSUPPORTED;
  const int64_t num_slots = static_cast<int64_t>(num_blocks) * block_size;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (head_dim == 128)
    e = launch_pdl(cache_write_fp8_kernel<128>, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
                   s, static_cast<const __nv_bfloat16*>(k_new),
                   static_cast<const __nv_bfloat16*>(v_new), slot_mapping, num_tokens,
                   static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), k_scale,
                   v_scale, num_slots, num_kv_heads, block_size,
                   static_cast<const int32_t*>(nullptr), static_cast<const int32_t*>(nullptr), 0);
  else
    e = launch_pdl(cache_write_fp8_kernel<64>, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
                   s, static_cast<const __nv_bfloat16*>(k_new),
                   static_cast<const __nv_bfloat16*>(v_new), slot_mapping, num_tokens,
                   static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), k_scale,
                   v_scale, num_slots, num_kv_heads, block_size,
                   static_cast<const int32_t*>(nullptr), static_cast<const int32_t*>(nullptr), 0);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_copy_blocks(void* k_cache, void* v_cache, float* k_scale,
                                    float* v_scale, const int32_t* pairs, int32_t num_pairs,
                                    int32_t num_blocks, int32_t num_kv_heads,
                                    int32_t block_size, int32_t head_dim,
                                    pa_kv_dtype kv_dtype, void* stream) {
  const NvtxRange nvtx_range("pa_copy_blocks");
  if (num_pairs < 0 || num_blocks < 0 || num_kv_heads <= 0 || block_size <= 0 || head_dim <= 0)
    return PA_ERR_INVALID_ARG;
  int esz;
  if (kv_dtype == PA_KV_BF16) {
    esz = 2;
  } else if (kv_dtype == PA_KV_FP8_E4M3) {
    esz = 1;
    if (num_pairs > 0 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  } else {
    return PA_ERR_INVALID_ARG;
  }
  if ((head_dim * esz) % 16 != 0) return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !pairs || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  if (num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  dim3 grid(static_cast<unsigned>(num_pairs), static_cast<unsigned>(num_kv_heads), 2);
  copy_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
      kv_dtype == PA_KV_FP8_E4M3 ? k_scale : nullptr,
      kv_dtype == PA_KV_FP8_E4M3 ? v_scale : nullptr, pairs, num_blocks, num_kv_heads,
      block_size, head_dim * esz / 16);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

namespace pa {
namespace {

// The address a kernel uses for a host buffer: pinned (page-locked or
// registered) or managed memory only.
bool host_device_ptr(const void* p, void** out) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type != cudaMemoryTypeHost && a.type != cudaMemoryTypeManaged) return false;
  *out = a.devicePointer != nullptr ? a.devicePointer : const_cast<void*>(p);
  return true;
}

pa_status swap_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                      const int32_t* block_ids, int32_t num_ids, void* host_k, void* host_v,
                      float* host_ks, float* host_vs, int32_t num_blocks, int32_t num_kv_heads,
                      int32_t block_size, int32_t head_dim, pa_kv_dtype kv_dtype, void* stream,
                      bool to_host) {
  if (num_ids < 0 || num_blocks < 0 || num_kv_heads <= 0 || block_size <= 0 || head_dim <= 0)
    return PA_ERR_INVALID_ARG;
  int esz;
  const bool fp8 = kv_dtype == PA_KV_FP8_E4M3;
  if (kv_dtype == PA_KV_BF16)
    esz = 2;
  else if (fp8)
    esz = 1;
  else
    return PA_ERR_INVALID_ARG;
  if ((head_dim * esz) % 16 != 0) return PA_ERR_INVALID_ARG;
  if (num_ids == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_ids || !host_k || !host_v || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(host_k) || !aligned16(host_v) ||
      (reinterpret_cast<uintptr_t>(block_ids) & 3u))
    return PA_ERR_INVALID_ARG;
  if (fp8 && (!k_scale || !v_scale || !host_ks || !host_vs)) return PA_ERR_INVALID_ARG;
  void *hk = nullptr, *hv = nullptr, *hks = nullptr, *hvs = nullptr;
  if (!host_device_ptr(host_k, &hk) || !host_device_ptr(host_v, &hv)) return PA_ERR_INVALID_ARG;
  if (fp8 && (!host_device_ptr(host_ks, &hks) || !host_device_ptr(host_vs, &hvs)))
    return PA_ERR_INVALID_ARG;
  int sms = 0;
  const pa_status st = device_sms(&sms, nullptr);
  if (st != PA_OK) return st;
  const int64_t block_chunks = static_cast<int64_t>(num_kv_heads) * block_size * head_dim * esz / 16;
  const int64_t total = 2 * block_chunks * num_ids;
  int64_t grid = (total + 4 * 256 - 1) / (4 * 256);
  if (grid > static_cast<int64_t>(sms) * 8) grid = static_cast<int64_t>(sms) * 8;
  if (grid < 1) grid = 1;
  return launch_pdl(swap_blocks_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
                    static_cast<cudaStream_t>(stream), static_cast<uint4*>(k_cache),
                    static_cast<uint4*>(v_cache), fp8 ? k_scale : nullptr,
                    fp8 ? v_scale : nullptr, static_cast<uint4*>(hk), static_cast<uint4*>(hv),
                    static_cast<float*>(hks), static_cast<float*>(hvs), block_ids, num_ids,
                    num_blocks, num_kv_heads, block_chunks, to_host) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_swap_out(const void* k_cache, const void* v_cache, const float* k_scale,
                                 const float* v_scale, const int32_t* block_ids, int32_t num_ids,
                                 void* host_k, void* host_v, float* host_k_scale,
                                 float* host_v_scale, int32_t num_blocks, int32_t num_kv_heads,
                                 int32_t block_size, int32_t head_dim, pa_kv_dtype kv_dtype,
                                 void* stream) {
  const NvtxRange nvtx_range("pa_swap_out");
  return swap_blocks(const_cast<void*>(k_cache), const_cast<void*>(v_cache),
                     const_cast<float*>(k_scale), const_cast<float*>(v_scale), block_ids,
                     num_ids, host_k, host_v, host_k_scale, host_v_scale, num_blocks,
                     num_kv_heads, block_size, head_dim, kv_dtype, stream, true);
}

extern "C" pa_status pa_swap_in(const void* host_k, const void* host_v,
                                const float* host_k_scale, const float* host_v_scale,
                                const int32_t* block_ids, int32_t num_ids, void* k_cache,
                                void* v_cache, float* k_scale, float* v_scale,
                                int32_t num_blocks, int32_t num_kv_heads, int32_t block_size,
                                int32_t head_dim, pa_kv_dtype kv_dtype, void* stream) {
  const NvtxRange nvtx_range("pa_swap_in");
  return swap_blocks(k_cache, v_cache, k_scale, v_scale, block_ids, num_ids,
                     const_cast<void*>(host_k), const_cast<void*>(host_v),
                     const_cast<float*>(host_k_scale), const_cast<float*>(host_v_scale),
                     num_blocks, num_kv_heads, block_size, head_dim, kv_dtype, stream, false);
}

extern "C" pa_status pa_quantize_fp8(const void* k_src, const void* v_src,
                                     const int32_t* block_ids, const int32_t* valid_lens,
                                     int32_t num_ids, uint8_t* k_dst, uint8_t* v_dst,
                                     float* k_scale, float* v_scale, int32_t num_blocks,
                                     int32_t num_kv_heads, int32_t block_size,
                                     int32_t head_dim, void* stream) {
  const NvtxRange nvtx_range("pa_quantize_fp8");
  if (num_ids < 0 || num_blocks < 0 || num_kv_heads <= 0 || block_size <= 0 ||
      head_dim <= 0 || head_dim % 16 != 0)
    return PA_ERR_INVALID_ARG;
  if (num_ids == 0) return PA_OK;
  if (!k_src || !v_src || !block_ids || !valid_lens || !k_dst || !v_dst || !k_scale || !v_scale)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(k_src) || !aligned16(v_src) || !aligned16(k_dst) || !aligned16(v_dst))
    return PA_ERR_INVALID_ARG;
  if (num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  dim3 grid(static_cast<unsigned>(num_ids), static_cast<unsigned>(num_kv_heads), 2);
  quantize_fp8_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_src), static_cast<const uint4*>(v_src), block_ids,
      valid_lens, reinterpret_cast<uint2*>(k_dst), reinterpret_cast<uint2*>(v_dst), k_scale,
      v_scale, num_blocks, num_kv_heads, block_size, head_dim);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

namespace {

pa_status auto_ctas(int32_t head_dim, pa_kv_dtype dt, int32_t* out) {
  int sms = 0, dev = 0;
  pa_status st = device_sms(&sms, &dev);
  if (st != PA_OK) return st;
  DecodePlan pl;
  if (dt == PA_KV_BF16 && head_dim == 128)
    st = decode_plan<128, false>(dev, &pl);
  else if (dt == PA_KV_BF16 && head_dim == 64)
    st = decode_plan<64, false>(dev, &pl);
  else if (dt == PA_KV_FP8_E4M3 && head_dim == 128)
    st = decode_plan<128, true>(dev, &pl);
  else if (dt == PA_KV_FP8_E4M3 && head_dim == 64)
    st = decode_plan<64, true>(dev, &pl);
  else if (dt == PA_KV_NVFP4)
    st = head_dim == 128 ? fp4_plan<128>(dev, &pl.ctas_per_sm) : fp4_plan<64>(dev, &pl.ctas_per_sm);
  else
    return PA_ERR_UNSUPPORTED;
  if (st != PA_OK) return st;
  const int per = pl.ctas_per_sm;
  *out = sms * per;
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                              int32_t num_kv_heads, int32_t head_dim,
                                              int32_t num_splits, size_t* bytes) {
  if (bytes == nullptr || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_splits < 0)
    return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  int32_t P = num_splits;
  if (P == 0) {
    // One size for every cache format: the largest automatic partition
    // count.
    int32_t a = 0, b = 0, c = 0;
    pa_status st = auto_ctas(head_dim, PA_KV_BF16, &a);
    if (st != PA_OK) return st;
    st = auto_ctas(head_dim, PA_KV_FP8_E4M3, &b);
    if (st != PA_OK) return st;
    st = auto_ctas(head_dim, PA_KV_NVFP4, &c);
    if (st != PA_OK) return st;
    P = a > b ? a : b;
    P = P > c ? P : c;
  }
  *bytes = P > 1 ? workspace_bytes_for(P, static_cast<int64_t>(num_seqs) * num_kv_heads,
                                       head_dim)
                 : 0;
  return PA_OK;
}

namespace pa {
namespace {

struct AppendArgs {
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
};

struct CascadeArgs {
  int32_t prefix_len;
  float* pf_o;
  float2* pf_ml;
  int32_t splits;
  int64_t stride;
};

// Token splits of the prefix pass: as many as one wave of CTAs (one per SM:
// each holds ~210 KB of shared memory and the tensor memory) allows, at
// least one chunk each, at most kPfMaxSplits (the merge holds them all in
// registers).
int32_t prefix_splits(int sms, int64_t num_seqs, int32_t group, int32_t num_kv_heads,
                      int32_t prefix_len) {
  const int64_t chunks = (prefix_len + kPfChunk - 1) / kPfChunk;
  const int64_t ctas = (num_seqs * group + kPfTiles * kPfRows - 1) / (kPfTiles * kPfRows) *
                       num_kv_heads;
  int64_t s = static_cast<int64_t>(sms) / ctas;
  if (s > chunks) s = chunks;
  if (s > kPfMaxSplits) s = kPfMaxSplits;
  if (s < 1) s = 1;
  return static_cast<int32_t>(s);
}

// Bytes of the prefix partials of a cascade (one per split and row; the
// merge folds them into split 0's), rounded up to 256.
size_t prefix_partial_bytes(int32_t splits, int64_t num_seqs, int32_t num_q_heads,
                            int32_t head_dim) {
  const size_t b = static_cast<size_t>(splits) * num_seqs * num_q_heads *
                   (static_cast<size_t>(head_dim) * sizeof(float) + sizeof(float2));
  return (b + 255) & ~static_cast<size_t>(255);
}

template <int D>
pa_status launch_prefix(const PrefixParams& pp, const void* k_cache, const void* v_cache,
                        cudaStream_t stream) {
  static bool attr_set[kMaxDevices] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(prefix_attention_kernel<D>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               PfSmem<D>::kBytes) != cudaSuccess)
        return PA_ERR_CUDA;
      attr_set[dev] = true;
    }
  }
  // K and V as 2D [rows][D] bf16, boxes of 64 columns x min(bs, 64) rows
  const int box_rows = pp.block_size < kPfChunk ? pp.block_size : kPfChunk;
  CUtensorMap tk, tv;
  if (!encode_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k_cache, D, pp.rows_total, D * 2, 64,
                 box_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v_cache, D, pp.rows_total, D * 2, 64,
                 box_rows, CU_TENSOR_MAP_SWIZZLE_128B))
    return PA_ERR_CUDA;
  const int64_t bx = (static_cast<int64_t>(pp.num_seqs) * pp.group + kPfTiles * kPfRows - 1) /
                     (kPfTiles * kPfRows);
  if (bx > INT_MAX || pp.num_kv_heads > 65535 || pp.splits > kPfMaxSplits) return PA_ERR_UNSUPPORTED;
  if (launch_pdl(prefix_attention_kernel<D>,
                 dim3(static_cast<unsigned>(bx), static_cast<unsigned>(pp.num_kv_heads),
                      static_cast<unsigned>(pp.splits)),
                 dim3(kPfThreads), PfSmem<D>::kBytes, stream, tk, tv, pp) != cudaSuccess)
    return PA_ERR_CUDA;
  if (pp.splits == 1) return PA_OK;
  // one partial per row for the suffix pass
  const int64_t threads = static_cast<int64_t>(pp.num_seqs) * pp.num_q_heads * (D / 4);
  const int64_t mx = (threads + 255) / 256;
  if (mx > INT_MAX) return PA_ERR_UNSUPPORTED;
  return launch_pdl(prefix_merge_kernel<D>, dim3(static_cast<unsigned>(mx)), dim3(256), 0,
                    stream, pp) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status decode_entry(const void* q, const void* k_cache, const void* v_cache,
                       const float* k_scale, const float* v_scale, pa_kv_dtype kv_dtype,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                       int32_t num_blocks, float scale, void* out, void* workspace,
                       size_t workspace_bytes, int32_t num_splits, void* stream,
                       const AppendArgs* app, const CascadeArgs* cas = nullptr) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq < 0 || num_splits < 0 || !(scale == scale) ||
      num_q_heads % num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
  const int32_t group = num_q_heads / num_kv_heads;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (group > kMaxG) return PA_ERR_UNSUPPORTED;
  if (!pow2_in(block_size, 8, 256)) return PA_ERR_UNSUPPORTED;
  // an FP8 append must find the whole block of the new token in the
  // sequence's last tile
  if (app != nullptr && kv_dtype == PA_KV_FP8_E4M3 && block_size > kTile)
    return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out) return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return PA_ERR_INVALID_ARG;
  if (app != nullptr &&
      (!app->k_new || !app->v_new || !app->slot_mapping || !aligned16(app->k_new) ||
       !aligned16(app->v_new) || (reinterpret_cast<uintptr_t>(app->slot_mapping) & 7u)))
    return PA_ERR_INVALID_ARG;
  if (kv_dtype == PA_KV_FP8_E4M3 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
  if (rows > INT_MAX - 64) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_seqs) * num_q_heads > INT_MAX - 64) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > INT_MAX - 64)
    return PA_ERR_UNSUPPORTED;

  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.block_size = block_size;
  p.log2_bs = ilog2(block_size);
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.rows_total = static_cast<int32_t>(rows);
  p.scale_log2 = scale * 1.4426950408889634f;
  if (cas != nullptr) {
    p.skip = cas->prefix_len;
    p.pf_o = cas->pf_o;
    p.pf_ml = cas->pf_ml;
  }
  if (app != nullptr) {
    p.k_new = static_cast<const uint8_t*>(app->k_new);
    p.v_new = static_cast<const uint8_t*>(app->v_new);
    p.slot_mapping = app->slot_mapping;
    p.k_cache = static_cast<uint8_t*>(const_cast<void*>(k_cache));
    p.v_cache = static_cast<uint8_t*>(const_cast<void*>(v_cache));
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kv_dtype == PA_KV_BF16) {
    if (head_dim == 128)
      return launch_decode<128, false>(p, q, k_cache, v_cache, workspace, workspace_bytes, num_splits, s);
    return launch_decode<64, false>(p, q, k_cache, v_cache, workspace, workspace_bytes, num_splits, s);
  }
  if (head_dim == 128 && cas == nullptr) {
    if (app != nullptr) {
      // FP8 append at head_dim 128: the checked cache write, then the
      // tcgen05 decode (its own launch: the decode kernel stores nothing)
      const int64_t warps = 2LL * num_seqs * num_kv_heads;
      const int64_t grid = (warps * 32 + 255) / 256;
      if (grid > INT_MAX) return PA_ERR_UNSUPPORTED;
      if (launch_pdl(cache_write_fp8_kernel<128>, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
                     s, static_cast<const __nv_bfloat16*>(app->k_new),
                     static_cast<const __nv_bfloat16*>(app->v_new), app->slot_mapping, num_seqs,
                     p.k_cache, p.v_cache, const_cast<float*>(k_scale),
                     const_cast<float*>(v_scale), static_cast<int64_t>(num_blocks) * block_size,
                     num_kv_heads, block_size, seq_lens, block_tables,
                     max_blocks_per_seq) != cudaSuccess)
        return PA_ERR_CUDA;
      p.k_new = p.v_new = nullptr;
      p.slot_mapping = nullptr;
      p.k_cache = p.v_cache = nullptr;
    }
    return launch_decode_tc<128>(p, q, k_cache, v_cache, workspace, workspace_bytes, num_splits,
                                 s);
  }
  if (head_dim == 128)
    return launch_decode<128, true>(p, q, k_cache, v_cache, workspace, workspace_bytes, num_splits, s);
  return launch_decode<64, true>(p, q, k_cache, v_cache, workspace, workspace_bytes, num_splits, s);
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale,
                               pa_kv_dtype kv_dtype, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* seq_lens,
                               int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int32_t num_blocks,
                               float scale, void* out, void* workspace,
                               size_t workspace_bytes, int32_t num_splits, void* stream) {
  const NvtxRange nvtx_range("pa_decode");
  return decode_entry(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, block_tables,
                      max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, scale, out, workspace, workspace_bytes,
                      num_splits, stream, nullptr);
}

extern "C" pa_status pa_decode_append_fp8(const void* q, const void* k_new, const void* v_new,
                                          const int64_t* slot_mapping, void* k_cache,
                                          void* v_cache, float* k_scale, float* v_scale,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* seq_lens, int32_t num_seqs,
                                          int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size,
                                          int32_t num_blocks, float scale, void* out,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t num_splits, void* stream) {
  const NvtxRange nvtx_range("pa_decode_append_fp8");
  const AppendArgs app{k_new, v_new, slot_mapping};
  return decode_entry(q, k_cache, v_cache, k_scale, v_scale, PA_KV_FP8_E4M3, block_tables,
                      max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, scale, out, workspace, workspace_bytes,
                      num_splits, stream, &app);
}

extern "C" pa_status pa_decode_append(const void* q, const void* k_new, const void* v_new,
                                      const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                      float scale, void* out, void* workspace,
                                      size_t workspace_bytes, int32_t num_splits, void* stream) {
  const NvtxRange nvtx_range("pa_decode_append");
  const AppendArgs app{k_new, v_new, slot_mapping};
  return decode_entry(q, k_cache, v_cache, nullptr, nullptr, PA_KV_BF16, block_tables,
                      max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, scale, out, workspace, workspace_bytes,
                      num_splits, stream, &app);
}

extern "C" pa_status pa_decode_cascade_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                                      int32_t num_kv_heads, int32_t head_dim,
                                                      int32_t block_size, int32_t prefix_len,
                                                      int32_t num_splits, size_t* bytes) {
  if (bytes == nullptr || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      block_size <= 0 || prefix_len < 0 || num_q_heads % num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  size_t dec = 0;
  const pa_status st = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                num_splits, &dec);
  if (st != PA_OK) return st;
  size_t pf = 0;
  if (prefix_len > 0 && num_seqs > 0) {
    int sms = 0;
    const pa_status s2 = device_sms(&sms, nullptr);
    if (s2 != PA_OK) return s2;
    const int32_t sp = prefix_splits(sms, num_seqs, num_q_heads / num_kv_heads, num_kv_heads,
                                     prefix_len);
    pf = prefix_partial_bytes(sp, num_seqs, num_q_heads, head_dim);
  }
  *bytes = pf + dec;
  return PA_OK;
}

extern "C" pa_status pa_decode_cascade(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                       int32_t prefix_len, float scale, void* out,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t num_splits, void* stream) {
  const NvtxRange nvtx_range("pa_decode_cascade");
  if (prefix_len < 0 || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      block_size <= 0 || max_blocks_per_seq < 0 || num_q_heads % num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  if (prefix_len % kTile != 0 || prefix_len % block_size != 0 ||
      static_cast<int64_t>(prefix_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
    return PA_ERR_INVALID_ARG;
  if (prefix_len == 0 || num_seqs == 0)
    return decode_entry(q, k_cache, v_cache, nullptr, nullptr, PA_KV_BF16, block_tables,
                        max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                        head_dim, block_size, num_blocks, scale, out, workspace,
                        workspace_bytes, num_splits, stream, nullptr);
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (num_q_heads / num_kv_heads > kMaxG) return PA_ERR_UNSUPPORTED;
  if (!pow2_in(block_size, 8, 256)) return PA_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !block_tables || !workspace || !aligned16(workspace) ||
      !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  if (!(scale == scale)) return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_blocks) * num_kv_heads * block_size > INT_MAX - 64)
    return PA_ERR_UNSUPPORTED;
  int sms = 0;
  pa_status st = device_sms(&sms, nullptr);
  if (st != PA_OK) return st;
  const int32_t group = num_q_heads / num_kv_heads;
  const int32_t sp = prefix_splits(sms, num_seqs, group, num_kv_heads, prefix_len);
  const size_t pf = prefix_partial_bytes(sp, num_seqs, num_q_heads, head_dim);
  if (workspace_bytes < pf) return PA_ERR_WORKSPACE;
  CascadeArgs cas;
  cas.prefix_len = prefix_len;
  cas.splits = 1;  // the prefix merge leaves one partial per row (split 0's slot)
  cas.stride = static_cast<int64_t>(num_seqs) * num_q_heads;
  cas.pf_o = static_cast<float*>(workspace);
  cas.pf_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) +
                                        static_cast<size_t>(sp) * cas.stride * head_dim *
                                            sizeof(float));
  PrefixParams pp;
  std::memset(&pp, 0, sizeof(pp));
  pp.q = static_cast<const uint8_t*>(q);
  pp.prefix_table = block_tables;  // sequence 0's row
  pp.pf_o = cas.pf_o;
  pp.pf_ml = cas.pf_ml;
  pp.num_seqs = num_seqs;
  pp.num_q_heads = num_q_heads;
  pp.num_kv_heads = num_kv_heads;
  pp.group = group;
  pp.block_size = block_size;
  pp.log2_bs = ilog2(block_size);
  pp.num_blocks = num_blocks;
  pp.rows_total = num_blocks * num_kv_heads * block_size;
  pp.prefix_tokens = prefix_len;
  pp.prefix_chunks = (prefix_len + kPfChunk - 1) / kPfChunk;
  pp.splits = sp;
  pp.scale_log2 = scale * 1.4426950408889634f;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = head_dim == 128 ? launch_prefix<128>(pp, k_cache, v_cache, s)
                       : launch_prefix<64>(pp, k_cache, v_cache, s);
  if (st != PA_OK) return st;
  return decode_entry(q, k_cache, v_cache, nullptr, nullptr, PA_KV_BF16, block_tables,
                      max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, scale, out,
                      static_cast<char*>(workspace) + pf, workspace_bytes - pf, num_splits,
                      stream, nullptr, &cas);
}

// ------------------------------------------------------------ no-alloc ---
// Scratch for pa_decode_noalloc: a file-scope device array, so the entry
// point needs no allocation.  In host code the symbol is only a host-side
// stand-in; the device address is looked up per device with
// cudaGetSymbolAddress (with that device current) and cached.
namespace pa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];
void* g_noalloc_addr[kMaxDevices] = {nullptr};
std::mutex g_noalloc_mu;

pa_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return PA_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                       const float* k_scale, const float* v_scale,
                                       pa_kv_dtype kv_dtype, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                       int32_t num_seqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim,
                                       int32_t block_size, int32_t num_blocks, float scale,
                                       void* out, int32_t num_splits, void* stream) {
  const NvtxRange nvtx_range("pa_decode_noalloc");
  void* scratch = nullptr;
  const pa_status st = pa::noalloc_scratch(&scratch);
  if (st != PA_OK) return st;
  // pa_decode validates the arguments first and returns PA_ERR_WORKSPACE,
  // enqueuing nothing, when this shape needs more than the array holds.
  return pa_decode(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, block_tables,
                   max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                   head_dim, block_size, num_blocks, scale, out, scratch,
                   PA_NOALLOC_SCRATCH_BYTES, num_splits, stream);
}

// ------------------------------------------------------------------ NVFP4
namespace pa {
namespace {

bool fp4_shape_ok(int32_t head_dim, int32_t block_size) {
  return (head_dim == 64 || head_dim == 128) && pow2_in(block_size, 16, 256);
}

bool finite_pos(float x) { return x > 0.f && x <= 3.402823466e38f; }

template <int D>
pa_status launch_fp4_decode(const DecodeParams& prm_in, const Fp4Args& f, void* workspace,
                            size_t workspace_bytes, int32_t num_splits, cudaStream_t stream) {
  int sms = 0, dev = 0;
  pa_status st = device_sms(&sms, &dev);
  if (st != PA_OK) return st;
  int per = 0;
  st = fp4_plan<D>(dev, &per);
  if (st != PA_OK) return st;
  const int32_t P = num_splits > 0 ? num_splits : sms * per;
  const int64_t segs = static_cast<int64_t>(prm_in.num_seqs) * prm_in.num_kv_heads;
  const size_t need = P > 1 ? workspace_bytes_for(P, segs, D) : 0;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
    return PA_ERR_WORKSPACE;
  DecodeParams prm = prm_in;
  prm.num_ctas = P;
  prm.seg_cost = kSegCostFp4;
  prm.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  prm.stall = g_wait_stall.load(std::memory_order_relaxed);
  prm.ws_o = nullptr;
  prm.ws_ml = nullptr;
  prm.ws_job = nullptr;
  if (need > 0) {
    const int64_t pieces = P + segs;
    char* w = static_cast<char*>(workspace);
    prm.ws_o = reinterpret_cast<float*>(w);
    w += static_cast<size_t>(pieces) * kMaxG * D * sizeof(float);
    prm.ws_ml = reinterpret_cast<float2*>(w);
    w += static_cast<size_t>(pieces) * kMaxG * sizeof(float2);
    prm.ws_job = reinterpret_cast<int2*>(w);
  }
  if (launch_pdl(f.slot_mapping != nullptr ? paged_decode_nvfp4_kernel<D, true>
                                           : paged_decode_nvfp4_kernel<D, false>,
                 dim3(static_cast<unsigned>(P)), dim3(32), fp4_smem_bytes<D>(), stream, prm,
                 f) != cudaSuccess)
    return PA_ERR_CUDA;
  if (launch_pdl(paged_decode_merge_kernel<D>, dim3(static_cast<unsigned>(P)),
                 dim3(prm.group * D / 4), 0, stream, prm) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_cache_write_nvfp4(const void* k_new, const void* v_new,
                                          const int64_t* slot_mapping, int32_t num_tokens,
                                          void* k_cache, void* v_cache, void* k_sf, void* v_sf,
                                          float k_gscale, float v_gscale, int32_t num_blocks,
                                          int32_t num_kv_heads, int32_t block_size,
                                          int32_t head_dim, void* stream) {
  const NvtxRange nvtx_range("pa_cache_write_nvfp4");
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || !finite_pos(k_gscale) ||
      !finite_pos(v_gscale))
    return PA_ERR_INVALID_ARG;
  if (!fp4_shape_ok(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !k_sf || !v_sf ||
      !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(k_sf) || !aligned16(v_sf) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PA_ERR_INVALID_ARG;
  int sms = 0;
  pa_status st = device_sms(&sms, nullptr);
  if (st != PA_OK) return st;
  const int64_t rows = 2LL * num_tokens * num_kv_heads;
  const int64_t want = (rows + 7) / 8;
  const unsigned grid = static_cast<unsigned>(want < sms * 16LL ? want : sms * 16LL);
  const int64_t num_slots = static_cast<int64_t>(num_blocks) * block_size;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* kn = static_cast<const __nv_bfloat16*>(k_new);
  auto* vn = static_cast<const __nv_bfloat16*>(v_new);
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
  auto* ks = static_cast<uint8_t*>(k_sf);
  auto* vs = static_cast<uint8_t*>(v_sf);
  cudaError_t e;
  if (head_dim == 128)
    e = launch_pdl(cache_write_nvfp4_kernel<128>, dim3(grid), dim3(256), 0, s, kn, vn,
                   slot_mapping, num_tokens, num_kv_heads, block_size, num_slots, kc, ks, vc, vs,
                   k_gscale, v_gscale);
  else
    e = launch_pdl(cache_write_nvfp4_kernel<64>, dim3(grid), dim3(256), 0, s, kn, vn,
                   slot_mapping, num_tokens, num_kv_heads, block_size, num_slots, kc, ks, vc, vs,
                   k_gscale, v_gscale);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

namespace pa {
namespace {

pa_status fp4_decode_entry(const void* q, const void* k_cache, const void* v_cache,
                           const void* k_sf, const void* v_sf, float k_gscale, float v_gscale,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                           int32_t num_blocks, float scale, void* out, void* workspace,
                           size_t workspace_bytes, int32_t num_splits, void* stream,
                           const AppendArgs* app) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq < 0 || num_splits < 0 || !(scale == scale) ||
      num_q_heads % num_kv_heads != 0 || !finite_pos(k_gscale) || !finite_pos(v_gscale))
    return PA_ERR_INVALID_ARG;
  const int32_t group = num_q_heads / num_kv_heads;
  if (!fp4_shape_ok(head_dim, block_size) || group > kMaxG) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !k_sf || !v_sf || !block_tables || !seq_lens || !out ||
      !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_sf) ||
      !aligned16(v_sf) || !aligned16(out) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return PA_ERR_INVALID_ARG;
  if (app != nullptr &&
      (!app->k_new || !app->v_new || !app->slot_mapping || !aligned16(app->k_new) ||
       !aligned16(app->v_new) || (reinterpret_cast<uintptr_t>(app->slot_mapping) & 7u)))
    return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_seqs) * num_q_heads > INT_MAX - 64) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > INT_MAX - 64)
    return PA_ERR_UNSUPPORTED;
  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.block_size = block_size;
  p.log2_bs = ilog2(block_size);
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.scale_log2 = scale * 1.4426950408889634f;
  // the merge kernel flags a new token of an empty sequence
  if (app != nullptr) p.slot_mapping = app->slot_mapping;
  Fp4Args f;
  std::memset(&f, 0, sizeof(f));
  f.q = static_cast<const __nv_bfloat16*>(q);
  f.k = static_cast<uint8_t*>(const_cast<void*>(k_cache));
  f.v = static_cast<uint8_t*>(const_cast<void*>(v_cache));
  f.k_sf = static_cast<uint8_t*>(const_cast<void*>(k_sf));
  f.v_sf = static_cast<uint8_t*>(const_cast<void*>(v_sf));
  f.k_gs = k_gscale;
  f.v_gs = v_gscale;
  if (app != nullptr) {
    f.k_new = static_cast<const __nv_bfloat16*>(app->k_new);
    f.v_new = static_cast<const __nv_bfloat16*>(app->v_new);
    f.slot_mapping = app->slot_mapping;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (head_dim == 128)
    return launch_fp4_decode<128>(p, f, workspace, workspace_bytes, num_splits, s);
  return launch_fp4_decode<64>(p, f, workspace, workspace_bytes, num_splits, s);
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_nvfp4(const void* q, const void* k_cache, const void* v_cache,
                                     const void* k_sf, const void* v_sf, float k_gscale,
                                     float v_gscale, const int32_t* block_tables,
                                     int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                     int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                     float scale, void* out, void* workspace,
                                     size_t workspace_bytes, int32_t num_splits, void* stream) {
  const NvtxRange nvtx_range("pa_decode_nvfp4");
  return fp4_decode_entry(q, k_cache, v_cache, k_sf, v_sf, k_gscale, v_gscale, block_tables,
                          max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                          head_dim, block_size, num_blocks, scale, out, workspace,
                          workspace_bytes, num_splits, stream, nullptr);
}

extern "C" pa_status pa_decode_append_nvfp4(
    const void* q, const void* k_new, const void* v_new, const int64_t* slot_mapping,
    void* k_cache, void* v_cache, void* k_sf, void* v_sf, float k_gscale, float v_gscale,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int32_t num_blocks, float scale, void* out, void* workspace,
    size_t workspace_bytes, int32_t num_splits, void* stream) {
  const NvtxRange nvtx_range("pa_decode_append_nvfp4");
  const AppendArgs app{k_new, v_new, slot_mapping};
  return fp4_decode_entry(q, k_cache, v_cache, k_sf, v_sf, k_gscale, v_gscale, block_tables,
                          max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                          head_dim, block_size, num_blocks, scale, out, workspace,
                          workspace_bytes, num_splits, stream, &app);
}
