// FP8 (E4M3) paged KV-cache write (cache_write.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "fp8mla.h"

namespace fp8mla {

struct CacheWriteArgs {
  const uint16_t* x;            // bf16 rows [n_tokens, h_kv, head_dim], token stride x_token_stride elements
  int64_t x_token_stride;
  const int32_t* slot_mapping;  // [n_tokens]
  int n_tokens, h_kv, head_dim, page_size, num_blocks;
  uint8_t* cache;               // E4M3 [num_blocks, h_kv, page_size, head_dim]
  const float* tensor_scale;    // per-tensor mode (device scalar), else null
  float* token_scales;          // per-row mode [num_blocks, h_kv, page_size], else null
};

// Lanes that share one row: the largest power of two <= min(32, head_dim / 8).
int cache_write_group_lanes(int head_dim);
fp8mla_status_t cache_write_entry(const CacheWriteArgs& a, cudaStream_t stream);
uint32_t cache_write_read_and_clear_status();

}  // namespace fp8mla
