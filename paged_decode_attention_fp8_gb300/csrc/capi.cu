// The C ABI: argument checks, TMA descriptor encoding (cached), launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "cache_write.h"
#include "fp8mla.h"
#include "gqa_decode.h"
#include "mla_decode.h"
#include "sparse_mla.h"

namespace fp8mla {
namespace {

// Stage timing of fp8mla_decode (a measurement aid, off by default): events
// recorded between the call's kernels, on the device of the last timed call.
struct StageTimer {
  std::mutex mu;
  bool enabled = false;
  bool timed = false;  // a call was timed since the last enable
  int device = -1;
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
};
StageTimer& stage_timer() {
  static StageTimer t;
  return t;
}
// Events of the current device (created on first use, re-created when the device changes).
bool stage_events(StageTimer& t) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (t.device == dev && t.ev[0] != nullptr) return true;
  for (cudaEvent_t& e : t.ev) {
    if (e != nullptr) cudaEventDestroy(e);
    e = nullptr;
  }
  t.device = dev;
  for (cudaEvent_t& e : t.ev)
    if (cudaEventCreate(&e) != cudaSuccess) return false;
  return true;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D byte view {inner, rows, pages} of a paged cache, one box per call.
bool encode_3d_bytes(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t pages,
                     uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {inner, rows, pages};
  const cuuint64_t strides[2] = {inner, inner * rows};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Small cache of the MLA cache's two descriptors, keyed by (pointer, pages, device).
struct MlaMaps {
  const void* base = nullptr;
  int pages = -1;
  int device = -1;
  CUtensorMap lat, rope;
};

std::mutex g_map_mu;
MlaMaps g_map_cache[8];
int g_map_next = 0;

bool mla_maps(const void* kv, int num_pages, CUtensorMap* lat, CUtensorMap* rope) {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (auto& e : g_map_cache)
    if (e.base == kv && e.pages == num_pages && e.device == dev) {
      *lat = e.lat;
      *rope = e.rope;
      return true;
    }
  MlaMaps m;
  m.base = kv;
  m.pages = num_pages;
  m.device = dev;
  if (!encode_3d_bytes(&m.lat, kv, kMlaD, kMlaPage, num_pages, 128, kMlaPage, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_3d_bytes(&m.rope, kv, kMlaD, kMlaPage, num_pages, 64, kMlaPage, CU_TENSOR_MAP_SWIZZLE_NONE))
    return false;
  g_map_cache[g_map_next] = m;
  g_map_next = (g_map_next + 1) % 8;
  *lat = m.lat;
  *rope = m.rope;
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace: [partial O | partial (m, l) | quantised Q (E4M3 hi term) | per-row Q scale]
struct MlaWorkspace {
  size_t o, ml, qbuf, qscale, total;
};

MlaWorkspace mla_workspace_layout(int b, int num_units) {
  const size_t slots = static_cast<size_t>(b) + num_units;
  MlaWorkspace w;
  w.o = 0;
  w.ml = w.o + round_up(slots * kMlaRows * kMlaDV * sizeof(uint16_t), 256);
  w.qbuf = w.ml + round_up(slots * kMlaRows * sizeof(float2), 256);
  w.qscale = w.qbuf + round_up(static_cast<size_t>(b) * kMlaQBytes, 256);
  w.total = w.qscale + round_up(static_cast<size_t>(b) * kMlaRows * sizeof(float), 256);
  return w;
}

fp8mla_status_t check_kv_dtype(fp8mla_kv_dtype_t t) {
  return t == FP8MLA_KV_E4M3 ? FP8MLA_OK : FP8MLA_ERR_UNSUPPORTED_DTYPE;
}

}  // namespace

// The two TMA descriptors of a dense MLA cache (both entry points use this one cached encoder).
bool mla_kv_maps(const void* kv, int num_pages, CUtensorMap* lat, CUtensorMap* rope) {
  return mla_maps(kv, num_pages, lat, rope);
}

}  // namespace fp8mla

using namespace fp8mla;

extern "C" {

fp8mla_status_t fp8mla_set_wait_test(int32_t fault_page, uint64_t wait_limit_ns) {
  if (fault_page < 0) return FP8MLA_ERR_INVALID_ARG;
  return mla_set_wait_test(fault_page, wait_limit_ns) == cudaSuccess ? FP8MLA_OK : FP8MLA_ERR_CUDA;
}

fp8mla_status_t fp8mla_get_wait_timeout_site(fp8mla_stream_t stream, uint32_t* where) {
  if (where == nullptr) return FP8MLA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8MLA_ERR_CUDA;
  mla_read_and_clear_timeout_site(where);
  return FP8MLA_OK;
}

const char* fp8mla_status_string(fp8mla_status_t s) {
  switch (s) {
    case FP8MLA_OK: return "ok";
    case FP8MLA_ERR_INVALID_ARG: return "invalid argument";
    case FP8MLA_ERR_UNSUPPORTED_DTYPE: return "unsupported KV cache encoding (only OCP E4M3 is accepted)";
    case FP8MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FP8MLA_ERR_CUDA: return "CUDA error";
    case FP8MLA_ERR_DEVICE: return "device-side error";
  }
  return "unknown status";
}

int fp8mla_metadata_units(int num_sms) { return num_sms / 2 > 1 ? num_sms / 2 : 1; }

size_t fp8mla_workspace_bytes(int b, int s_q, int h_q, int num_units) {
  (void)s_q;
  (void)h_q;
  if (b < 0 || num_units < 1) return 0;
  return mla_workspace_layout(b, num_units).total;
}

fp8mla_status_t fp8mla_get_metadata(const int32_t* cache_seqlens, int b, int h_q, int s_q, int num_units,
                                    int force_splits, int32_t* tile_sched, int32_t* num_splits,
                                    fp8mla_stream_t stream) {
  if (b < 0 || h_q < 1 || s_q < 1 || h_q * s_q > kMlaRows || num_units < 1 || force_splits < 0)
    return FP8MLA_ERR_INVALID_ARG;
  if ((b > 0 && cache_seqlens == nullptr) || tile_sched == nullptr || num_splits == nullptr)
    return FP8MLA_ERR_INVALID_ARG;
  if (force_splits > 0 && static_cast<long long>(b) * force_splits > num_units) return FP8MLA_ERR_INVALID_ARG;
  if (metadata_smem_bytes(b, num_units) > kMetadataMaxSmem) return FP8MLA_ERR_INVALID_ARG;
  if (launch_mla_metadata(cache_seqlens, b, num_units, force_splits, tile_sched, num_splits,
                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FP8MLA_ERR_CUDA;
  return FP8MLA_OK;
}

}  // extern "C"

namespace fp8mla {
namespace {
// fp8mla_decode and fp8mla_decode_ext: kv_rows non-null = per-row scales [num_pages, 64].
fp8mla_status_t mla_decode_call(const void* q, const void* kv_cache, fp8mla_kv_dtype_t kv_dtype, int num_pages,
                                const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                                const float* kv_scale, const float* kv_rows, float softmax_scale, int causal,
                                const int32_t* tile_sched, const int32_t* num_splits, int num_units, void* workspace,
                                size_t workspace_bytes, void* out, float* lse, fp8mla_dot_mode_t dot_mode, int b,
                                int s_q, int h_q, fp8mla_stream_t stream) {
  fp8mla_status_t st = check_kv_dtype(kv_dtype);
  if (st != FP8MLA_OK) return st;
  if (b < 0 || s_q < 1 || h_q < 1 || s_q * h_q > kMlaRows || num_units < 1 || num_pages < 1 || max_pages < 1)
    return FP8MLA_ERR_INVALID_ARG;
  if (dot_mode != FP8MLA_DOT_FP8 && dot_mode != FP8MLA_DOT_16BIT) return FP8MLA_ERR_INVALID_ARG;
  if (kv_scale == nullptr && kv_rows == nullptr) return FP8MLA_ERR_INVALID_ARG;  // an FP8 cache without its scale
  // per-row scales: FP8 dots only, arriving by 256-byte bulk copies
  if (kv_rows != nullptr && (dot_mode != FP8MLA_DOT_FP8 || !aligned(kv_rows, 16))) return FP8MLA_ERR_INVALID_ARG;
  if (b == 0) return FP8MLA_OK;
  if (q == nullptr || kv_cache == nullptr || block_table == nullptr || cache_seqlens == nullptr ||
      tile_sched == nullptr || num_splits == nullptr || out == nullptr || lse == nullptr || workspace == nullptr)
    return FP8MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(workspace, 256))
    return FP8MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f)) return FP8MLA_ERR_INVALID_ARG;
  if (workspace_bytes < fp8mla_workspace_bytes(b, s_q, h_q, num_units)) return FP8MLA_ERR_WORKSPACE_TOO_SMALL;

  CUtensorMap tm_lat, tm_rope;
  if (!mla_maps(kv_cache, num_pages, &tm_lat, &tm_rope)) return FP8MLA_ERR_CUDA;

  const MlaWorkspace wl = mla_workspace_layout(b, num_units);
  char* ws = static_cast<char*>(workspace);
  MlaParams prm{};
  prm.q = static_cast<const uint16_t*>(q);
  prm.block_table = block_table;
  prm.seqlens = cache_seqlens;
  prm.kv_scale = kv_scale;
  prm.kv_rows = kv_rows;
  prm.tile_sched = tile_sched;
  prm.num_splits = num_splits;
  prm.ws_o = reinterpret_cast<uint16_t*>(ws + wl.o);
  prm.ws_ml = reinterpret_cast<float2*>(ws + wl.ml);
  prm.qbuf = reinterpret_cast<uint8_t*>(ws + wl.qbuf);
  prm.qscale = reinterpret_cast<float*>(ws + wl.qscale);
  prm.out = static_cast<uint16_t*>(out);
  prm.lse = lse;
  prm.softmax_scale = softmax_scale;
  prm.causal = causal ? 1 : 0;
  prm.max_pages = max_pages;
  prm.num_pages = num_pages;
  prm.b = b;
  prm.s_q = s_q;
  prm.h_q = h_q;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  StageTimer& timer = stage_timer();
  std::unique_lock<std::mutex> timing(timer.mu, std::defer_lock);
  bool timed = false;
  {
    std::lock_guard<std::mutex> g(timer.mu);
    timed = timer.enabled;
  }
  if (timed) {
    timing.lock();
    if (!stage_events(timer)) return FP8MLA_ERR_CUDA;
  }
  auto mark = [&](int i) { return timed ? cudaEventRecord(timer.ev[i], s) : cudaSuccess; };
  cudaError_t e = mark(0);
  if (e == cudaSuccess) e = launch_mla_qprep(prm, s);
  if (e == cudaSuccess) e = mark(1);
  if (e == cudaSuccess)
    e = (dot_mode == FP8MLA_DOT_FP8) ? launch_mla_decode_fp8(tm_lat, tm_rope, prm, num_units, s)
                                     : launch_mla_decode_16bit(tm_lat, tm_rope, prm, num_units, s);
  if (e == cudaSuccess) e = mark(2);
  if (e == cudaSuccess)
    e = launch_mla_combine(num_splits, prm.ws_o, prm.ws_ml, prm.q, prm.qscale, dot_mode == FP8MLA_DOT_16BIT,
                           softmax_scale, prm.out, lse, b, s_q * h_q, s);
  if (e == cudaSuccess) e = mark(3);
  if (e != cudaSuccess) return FP8MLA_ERR_CUDA;
  if (timed) timer.timed = true;
  return FP8MLA_OK;
}
}  // namespace
}  // namespace fp8mla

extern "C" {

fp8mla_status_t fp8mla_decode(const void* q, const void* kv_cache, fp8mla_kv_dtype_t kv_dtype, int num_pages,
                              const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                              const float* kv_scale, float softmax_scale, int causal, const int32_t* tile_sched,
                              const int32_t* num_splits, int num_units, void* workspace, size_t workspace_bytes,
                              void* out, float* lse, fp8mla_dot_mode_t dot_mode, int b, int s_q, int h_q,
                              fp8mla_stream_t stream) {
  if (kv_scale == nullptr && check_kv_dtype(kv_dtype) == FP8MLA_OK) return FP8MLA_ERR_INVALID_ARG;
  return mla_decode_call(q, kv_cache, kv_dtype, num_pages, block_table, max_pages, cache_seqlens, kv_scale, nullptr,
                         softmax_scale, causal, tile_sched, num_splits, num_units, workspace, workspace_bytes, out,
                         lse, dot_mode, b, s_q, h_q, stream);
}

fp8mla_status_t fp8mla_decode_ext(const void* q, const void* kv_cache, fp8mla_kv_dtype_t kv_dtype, int num_pages,
                                  const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                                  const float* kv_scale, const float* kv_scale_rows, float softmax_scale, int causal,
                                  const int32_t* tile_sched, const int32_t* num_splits, int num_units, void* workspace,
                                  size_t workspace_bytes, void* out, float* lse, fp8mla_dot_mode_t dot_mode, int b,
                                  int s_q, int h_q, fp8mla_stream_t stream) {
  return mla_decode_call(q, kv_cache, kv_dtype, num_pages, block_table, max_pages, cache_seqlens, kv_scale,
                         kv_scale_rows, softmax_scale, causal, tile_sched, num_splits, num_units, workspace,
                         workspace_bytes, out, lse, dot_mode, b, s_q, h_q, stream);
}

fp8mla_status_t fp8mla_set_stage_timing(int enable) {
  StageTimer& t = stage_timer();
  std::lock_guard<std::mutex> g(t.mu);
  t.enabled = enable != 0;
  t.timed = false;
  return FP8MLA_OK;
}

fp8mla_status_t fp8mla_get_stage_times(fp8mla_stream_t stream, float* ms) {
  if (ms == nullptr) return FP8MLA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8MLA_ERR_CUDA;
  StageTimer& t = stage_timer();
  std::lock_guard<std::mutex> g(t.mu);
  if (!t.timed) return FP8MLA_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i)
    if (cudaEventElapsedTime(&ms[i], t.ev[i], t.ev[i + 1]) != cudaSuccess) return FP8MLA_ERR_CUDA;
  return FP8MLA_OK;
}

size_t sparse_mla_workspace_bytes(int s_q, int h_q, int topk, int num_splits) {
  return sparse_workspace_bytes(s_q, h_q, topk, num_splits);
}

fp8mla_status_t sparse_mla_decode(const void* q, const void* kv_cache, fp8mla_kv_dtype_t kv_dtype,
                                  int64_t num_tokens, const int32_t* topk_idx, int topk, const float* kv_scale,
                                  float softmax_scale, int num_splits, void* workspace, size_t workspace_bytes,
                                  void* out, float* lse, fp8mla_dot_mode_t dot_mode, int s_q, int h_q,
                                  fp8mla_stream_t stream) {
  fp8mla_status_t st = check_kv_dtype(kv_dtype);
  if (st != FP8MLA_OK) return st;
  if (kv_scale == nullptr) return FP8MLA_ERR_INVALID_ARG;
  return sparse_decode_entry(q, kv_cache, num_tokens, topk_idx, topk, kv_scale, softmax_scale, num_splits,
                             workspace, workspace_bytes, out, lse, dot_mode, s_q, h_q,
                             reinterpret_cast<cudaStream_t>(stream));
}

size_t paged_gqa_workspace_bytes(int bs, int h_q, int head_dim, int max_splits) {
  return gqa_workspace_bytes(bs, h_q, head_dim, max_splits);
}

int paged_gqa_num_splits(int bs, int h_kv, int max_seqlen, int num_sms, int num_splits) {
  return gqa_choose_splits(bs, h_kv, max_seqlen, num_sms, num_splits);
}

int paged_gqa_ext_num_splits(int bs, int h_kv, int max_seqlen, int q_len, int window, int num_sms, int num_splits) {
  long long longest = max_seqlen;
  if (window > 0) longest = std::min(longest, static_cast<long long>(window) + std::max(q_len, 1) - 1 + 128);
  return gqa_choose_splits(bs, h_kv, static_cast<int>(longest), num_sms, num_splits, window > 0);
}

fp8mla_status_t paged_gqa_decode(const void* q, const void* k_cache, const void* v_cache,
                                 fp8mla_kv_dtype_t kv_dtype, int num_blocks, const float* k_scale,
                                 const float* v_scale, const int32_t* block_table, int max_blocks,
                                 const int32_t* seqlens, float softmax_scale, int num_splits, void* workspace,
                                 size_t workspace_bytes, void* out, float* lse, int bs, int h_q, int h_kv,
                                 int head_dim, int page_size, fp8mla_stream_t stream) {
  fp8mla_status_t st = check_kv_dtype(kv_dtype);
  if (st != FP8MLA_OK) return st;
  if (k_scale == nullptr || v_scale == nullptr) return FP8MLA_ERR_INVALID_ARG;
  return gqa_decode_entry(q, k_cache, v_cache, num_blocks, k_scale, v_scale, 0, block_table, max_blocks, seqlens,
                          softmax_scale, 1, nullptr, 0, nullptr, num_splits, workspace, workspace_bytes, out, lse, bs,
                          h_q, h_kv, head_dim, page_size, reinterpret_cast<cudaStream_t>(stream));
}

fp8mla_status_t paged_gqa_decode_ext(const void* q, const void* k_cache, const void* v_cache,
                                     fp8mla_kv_dtype_t kv_dtype, int num_blocks, const float* k_scale,
                                     const float* v_scale, int scale_per_row, const int32_t* block_table,
                                     int max_blocks, const int32_t* seqlens, float softmax_scale, int q_len,
                                     const uint8_t* spec_mask, int window, const float* sinks, int num_splits,
                                     void* workspace, size_t workspace_bytes, void* out, float* lse, int bs, int h_q,
                                     int h_kv, int head_dim, int page_size, fp8mla_stream_t stream) {
  fp8mla_status_t st = check_kv_dtype(kv_dtype);
  if (st != FP8MLA_OK) return st;
  if (k_scale == nullptr || v_scale == nullptr) return FP8MLA_ERR_INVALID_ARG;
  return gqa_decode_entry(q, k_cache, v_cache, num_blocks, k_scale, v_scale, scale_per_row, block_table, max_blocks,
                          seqlens, softmax_scale, q_len, spec_mask, window, sinks, num_splits, workspace,
                          workspace_bytes, out, lse, bs, h_q, h_kv, head_dim, page_size,
                          reinterpret_cast<cudaStream_t>(stream));
}

fp8mla_status_t fp8_paged_cache_write(const void* x, int64_t x_token_stride, const int32_t* slot_mapping,
                                      int n_tokens, int h_kv, int head_dim, int page_size, int num_blocks,
                                      fp8mla_kv_dtype_t kv_dtype, void* cache, const float* tensor_scale,
                                      float* token_scales, fp8mla_stream_t stream) {
  fp8mla_status_t st = check_kv_dtype(kv_dtype);
  if (st != FP8MLA_OK) return st;
  CacheWriteArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.x_token_stride = x_token_stride;
  a.slot_mapping = slot_mapping;
  a.n_tokens = n_tokens;
  a.h_kv = h_kv;
  a.head_dim = head_dim;
  a.page_size = page_size;
  a.num_blocks = num_blocks;
  a.cache = static_cast<uint8_t*>(cache);
  a.tensor_scale = tensor_scale;
  a.token_scales = token_scales;
  return cache_write_entry(a, reinterpret_cast<cudaStream_t>(stream));
}

fp8mla_status_t fp8mla_get_last_device_error(fp8mla_stream_t stream, uint32_t* code_out) {
  if (code_out == nullptr) return FP8MLA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8MLA_ERR_CUDA;
  *code_out = mla_read_and_clear_status() | metadata_read_and_clear_status() |
              sparse_read_and_clear_status() | gqa_read_and_clear_status() |
              cache_write_read_and_clear_status();
  return FP8MLA_OK;
}

}  // extern "C"
