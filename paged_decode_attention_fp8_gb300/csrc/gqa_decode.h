// Paged GQA decode with split-KV (gqa_decode.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "fp8mla.h"

namespace fp8mla {

size_t gqa_workspace_bytes(int bs, int h_q, int head_dim, int max_splits);
// capped: a sliding window bounds every sequence's keys (pieces need no balancing: a
// grid that fills the GPU is not split)
int gqa_choose_splits(int bs, int h_kv, int max_seqlen, int num_sms, int num_splits, bool capped = false);
// q_len query tokens per sequence (the last q_len cache positions) under spec_mask
// [bs, q_len, q_len] (null: causal inside the block), a sliding window (0: off) and
// sink logits [h_q] (null: none); scale_rows: k_scale / v_scale per cached row
// [num_blocks, h_kv, page] instead of [1].
fp8mla_status_t gqa_decode_entry(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                 const float* k_scale, const float* v_scale, int scale_rows,
                                 const int32_t* block_table, int max_blocks, const int32_t* seqlens,
                                 float softmax_scale, int q_len, const uint8_t* spec_mask, int window,
                                 const float* sinks, int num_splits, void* workspace, size_t workspace_bytes,
                                 void* out, float* lse, int bs, int h_q, int h_kv, int head_dim, int page_size,
                                 cudaStream_t stream);
uint32_t gqa_read_and_clear_status();

}  // namespace fp8mla
