// Host-side declarations shared by the C ABI and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fp8mla {

struct MlaParams {
  const uint16_t* q;           // bf16 [b, s_q, h_q, 576]
  const int32_t* block_table;  // [b, max_pages]
  const int32_t* seqlens;      // [b]
  const float* kv_scale;       // [1]
  const float* kv_rows;        // per-row scales [num_pages, 64] or null (FP8 dots only)
  const int32_t* tile_sched;   // [num_units, 8]
  const int32_t* num_splits;   // [b + 1]
  uint16_t* ws_o;              // [slots, 128, 512] partial accumulators as bf16 (true units)
  float2* ws_ml;               // [slots, 128] (m in log2 units, l)
  uint8_t* qbuf;               // [b, kMlaQBytes] Q quantised to E4M3 (its hi term for 16-bit dots), in the kernel's slot layout
  float* qscale;               // [b, 128] per-row power-of-two Q scale
  uint16_t* out;               // bf16 [b, s_q, h_q, 512]
  float* lse;                  // [b, s_q, h_q]
  float softmax_scale;
  int causal;
  int max_pages;
  int num_pages;
  int b, s_q, h_q;
};

constexpr int kMlaRows = 128;
constexpr int kMlaDV = 512;
constexpr int kMlaPage = 64;
constexpr int kMlaD = 576;
constexpr int kSchedFixedCost = 4;
// One sequence's quantised Q, in the decode kernel's ring-slot layout (two
// latent slots of 128 x 272 bytes, one RoPE slot of 128 x 144 bytes).
constexpr int kMlaQBytes = 88064;
constexpr size_t kMetadataMaxSmem = 200 * 1024;  // the scheduler stages ~16 bytes per sequence and unit
size_t metadata_smem_bytes(int b, int num_units);

// dense MLA decode kernels (mla_decode.cu): FP8 dots (per-tensor or per-row
// scales), 16-bit dots as two-term E4M3 dots (per-tensor scale)
cudaError_t launch_mla_decode_fp8(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const MlaParams& prm,
                                  int num_units, cudaStream_t stream);
cudaError_t launch_mla_decode_16bit(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const MlaParams& prm,
                                    int num_units, cudaStream_t stream);
uint32_t mla_read_and_clear_status();
// The TMA descriptors of a dense MLA cache [num_pages, 64, 576] E4M3: 128-byte latent boxes
// (128-byte swizzle) and the 64-byte RoPE box, cached per (pointer, pages, device).
bool mla_kv_maps(const void* kv, int num_pages, CUtensorMap* lat, CUtensorMap* rope);
// {source line, block, thread} of the first bounded wait of the dense MLA kernels that ran
// out since the last call (all 0 if none), and clears it.
void mla_read_and_clear_timeout_site(uint32_t where[3]);
// Test hook of the bounded waits of the FP8-dots MLA kernel on the current device:
// fault_page = p + 1 makes CTA 0 of work unit 0 skip the loads of its p-th page
// (0 = off); wait_limit_ns replaces the wait limit (0 = the default).
cudaError_t mla_set_wait_test(int fault_page, uint64_t wait_limit_ns);
// Quantises every sequence's Q rows into prm.qbuf / prm.qscale (launched
// right before the decode kernel of either dot mode, as a programmatic dependent).
cudaError_t launch_mla_qprep(const MlaParams& prm, cudaStream_t stream);

// metadata + combine (metadata.cu)
cudaError_t launch_mla_metadata(const int32_t* seqlens, int b, int num_units, int force_splits, int32_t* tile_sched,
                                int32_t* num_splits, cudaStream_t stream);
// Merges split partials into out / lse, and (q, the bf16 queries, and qscale,
// their per-row power-of-two scales, non-null) applies the first-order
// Q-quantisation correction to every row's LSE from the finished output row
// and q_hat - q, recomputed with the decode kernel's rounding: one E4M3 term
// (FP8 dots) or two (two_term, 16-bit dots).
cudaError_t launch_mla_combine(const int32_t* num_splits, const uint16_t* ws_o, const float2* ws_ml,
                               const uint16_t* q, const float* qscale, bool two_term, float softmax_scale,
                               uint16_t* out, float* lse, int b, int rows, cudaStream_t stream);
uint32_t metadata_read_and_clear_status();

}  // namespace fp8mla
