// fp8mla_decode_no_alloc: the dense MLA decode for callers that cannot
// allocate device memory.  It needs the same scratch as fp8mla_decode (a
// tile schedule, split counts, the per-row LSE-correction terms and, for FP8
// dots, the quantised Q with its per-row scales), but
// takes it from a fixed array that lives in this library instead of from the
// caller.  It schedules one work unit per sequence (no split-KV), so the
// split partials of fp8mla_decode's workspace are never used.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fp8mla.h"
#include "mla_decode.h"

namespace fp8mla {
namespace {

constexpr int kNoAllocMaxBatch = FP8MLA_NO_ALLOC_MAX_BATCH;
constexpr size_t kSchedBytes = 256 * 8 * sizeof(int32_t);                         // tile schedule, <= 256 units
constexpr size_t kSplitsBytes = 256 * sizeof(int32_t);                            // split prefix, <= 255 sequences
constexpr size_t kQBufBytes = static_cast<size_t>(kNoAllocMaxBatch) * kMlaQBytes;    // quantised Q
constexpr size_t kQScaleBytes = static_cast<size_t>(kNoAllocMaxBatch) * kMlaRows * sizeof(float);
constexpr size_t kScratchBytes = kSchedBytes + kSplitsBytes + kQBufBytes + kQScaleBytes;  // 5.7 MB
static_assert(kNoAllocMaxBatch <= 255, "the split prefix holds b + 1 entries");

// Held by every GPU that loads the library, for the life of the process.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kScratchBytes];

// Device address of the array, looked up once per device with that device current.
std::mutex g_mu;
void* g_scratch_ptr[64] = {};

void* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace fp8mla

using namespace fp8mla;

extern "C" fp8mla_status_t fp8mla_decode_no_alloc(const void* q, const void* kv_cache, fp8mla_kv_dtype_t kv_dtype,
                                                  int num_pages, const int32_t* block_table, int max_pages,
                                                  const int32_t* cache_seqlens, const float* kv_scale,
                                                  float softmax_scale, int causal, void* out, float* lse,
                                                  fp8mla_dot_mode_t dot_mode, int b, int s_q, int h_q,
                                                  fp8mla_stream_t stream) {
  if (kv_dtype != FP8MLA_KV_E4M3) return FP8MLA_ERR_UNSUPPORTED_DTYPE;
  if (b < 0 || s_q < 1 || h_q < 1 || s_q * h_q > kMlaRows || num_pages < 1 || max_pages < 1 ||
      !(softmax_scale > 0.f) || (dot_mode != FP8MLA_DOT_FP8 && dot_mode != FP8MLA_DOT_16BIT) || kv_scale == nullptr)
    return FP8MLA_ERR_INVALID_ARG;
  if (b > kNoAllocMaxBatch) return FP8MLA_ERR_WORKSPACE_TOO_SMALL;  // beyond the fixed array's capacity
  if (b == 0) return FP8MLA_OK;
  if (q == nullptr || kv_cache == nullptr || block_table == nullptr || cache_seqlens == nullptr || out == nullptr ||
      lse == nullptr)
    return FP8MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_cache) | reinterpret_cast<uintptr_t>(out)) &
      15u)
    return FP8MLA_ERR_INVALID_ARG;

  unsigned char* scratch = static_cast<unsigned char*>(scratch_for_current_device());
  if (scratch == nullptr) return FP8MLA_ERR_CUDA;
  int32_t* tile_sched = reinterpret_cast<int32_t*>(scratch);
  int32_t* num_splits = reinterpret_cast<int32_t*>(scratch + kSchedBytes);
  uint8_t* qbuf = reinterpret_cast<uint8_t*>(scratch) + kSchedBytes + kSplitsBytes;
  float* qscale = reinterpret_cast<float*>(qbuf + kQBufBytes);

  CUtensorMap tm_lat, tm_rope;
  if (!mla_kv_maps(kv_cache, num_pages, &tm_lat, &tm_rope)) return FP8MLA_ERR_CUDA;

  // One unit per sequence: every sequence is one whole piece, so the split
  // partials (ws_o, ws_ml) are never written or read.  The schedule and the
  // quantised Q are rewritten by every call before they are read, so nothing
  // left in the array by an earlier call needs clearing.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int units = b;
  if (launch_mla_metadata(cache_seqlens, b, units, 1, tile_sched, num_splits, s) != cudaSuccess)
    return FP8MLA_ERR_CUDA;
  MlaParams prm{};
  prm.q = static_cast<const uint16_t*>(q);
  prm.block_table = block_table;
  prm.seqlens = cache_seqlens;
  prm.kv_scale = kv_scale;
  prm.kv_rows = nullptr;  // per-tensor scale only
  prm.tile_sched = tile_sched;
  prm.num_splits = num_splits;
  prm.ws_o = nullptr;
  prm.ws_ml = nullptr;
  prm.qbuf = qbuf;
  prm.qscale = qscale;
  prm.out = static_cast<uint16_t*>(out);
  prm.lse = lse;
  prm.softmax_scale = softmax_scale;
  prm.causal = causal ? 1 : 0;
  prm.max_pages = max_pages;
  prm.num_pages = num_pages;
  prm.b = b;
  prm.s_q = s_q;
  prm.h_q = h_q;
  cudaError_t e = launch_mla_qprep(prm, s);
  if (e == cudaSuccess)
    e = (dot_mode == FP8MLA_DOT_FP8) ? launch_mla_decode_fp8(tm_lat, tm_rope, prm, units, s)
                                     : launch_mla_decode_16bit(tm_lat, tm_rope, prm, units, s);
  if (e != cudaSuccess) return FP8MLA_ERR_CUDA;
  if (launch_mla_combine(num_splits, nullptr, nullptr, prm.q, qscale, dot_mode == FP8MLA_DOT_16BIT, softmax_scale,
                         prm.out, lse, b, s_q * h_q, s) != cudaSuccess)
    return FP8MLA_ERR_CUDA;
  return FP8MLA_OK;
}
