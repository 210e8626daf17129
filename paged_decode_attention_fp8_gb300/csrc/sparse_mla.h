// Top-k sparse MLA decode (sparse_mla.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "fp8mla.h"

namespace fp8mla {

size_t sparse_workspace_bytes(int s_q, int h_q, int topk, int num_splits);
fp8mla_status_t sparse_decode_entry(const void* q, const void* kv_cache, int64_t num_tokens, const int32_t* topk_idx,
                                    int topk, const float* kv_scale, float softmax_scale, int num_splits,
                                    void* workspace, size_t workspace_bytes, void* out, float* lse,
                                    fp8mla_dot_mode_t dot_mode, int s_q, int h_q, cudaStream_t stream);
uint32_t sparse_read_and_clear_status();

}  // namespace fp8mla
