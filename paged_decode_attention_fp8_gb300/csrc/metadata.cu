// Tile scheduling for the dense MLA kernel and the split-KV combine kernel.
//
// Scheduling: the flattened (sequence, 64-token page) work list is cut into
// num_units contiguous ranges.  Each page costs 1 and each (sequence, unit)
// piece a fixed kSchedFixedCost more (Q load + epilogue).  A unit's budget is
// ceil(total / num_units) + fixed; it takes whole remainders of sequences
// while they fit, else (budget left - fixed) pages of the current one, and
// the last unit takes what is left.  A sequence cut across units becomes
// several splits whose partial (m, l, acc) the combine kernel merges: the
// split-KV flash-decoding of the InfiniCore "FP8(E4M3) KV cache support in
// paged attention" page (split-kv commit), with a balanced persistent
// schedule instead of a fixed split count.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "mla_decode.h"

namespace fp8mla {

__device__ uint32_t g_status_meta;

namespace {

__device__ __forceinline__ int pages_of(int s_k) {
  if (s_k < 0) atomicOr(&g_status_meta, FP8MLA_DEV_BAD_SEQLEN);
  return s_k > 0 ? (s_k + kMlaPage - 1) / kMlaPage : 0;
}

__device__ __forceinline__ void put_row(int32_t* row, int a, int b, int c, int d, int e) {
  row[0] = a;
  row[1] = b;
  row[2] = c;
  row[3] = d;
  row[4] = e;
  row[5] = 0;
  row[6] = 0;
  row[7] = 0;
}

// One warp stages the page counts in shared memory; lane 0 then runs the
// sequential rule (it touches b + num_units items) at shared-memory latency.
__global__ void mla_metadata_kernel(const int32_t* __restrict__ seqlens, int B, int U, int force,
                                    int32_t* __restrict__ sched, int32_t* __restrict__ num_splits) {
  extern __shared__ int32_t meta_smem[];
  int32_t* n = meta_smem;        // pages per sequence
  int32_t* count = n + B;        // splits per sequence
  if (blockIdx.x != 0) return;
  for (int i = threadIdx.x; i < B; i += blockDim.x) {
    n[i] = pages_of(seqlens[i]);
    count[i] = 0;
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    if (force > 0) {
      int u = 0;
      for (int bi = 0; bi < B; ++bi) {
        const int nb = n[bi];
        const int c = min(force, nb);
        for (int j = 0; j < c; ++j, ++u) {
          if (u >= U) continue;  // the host refuses b * force > num_units
          const int p0 = static_cast<int>((static_cast<long long>(j) * nb) / c);
          const int p1 = static_cast<int>((static_cast<long long>(j + 1) * nb) / c);
          if (p1 == nb)
            put_row(sched + 8 * u, bi, p0, bi + 1, 0, j);
          else
            put_row(sched + 8 * u, bi, p0, bi, p1, j);
          count[bi] += 1;
        }
      }
      for (; u < U; ++u) put_row(sched + 8 * u, B, 0, B, 0, 0);
    } else {
      long long total = 0;
      for (int bi = 0; bi < B; ++bi)
        if (n[bi] > 0) total += n[bi] + kSchedFixedCost;
      const long long budget = total > 0 ? (total + U - 1) / U + kSchedFixedCost : 0;
      int bi = 0, p = 0;
      for (int u = 0; u < U; ++u) {
        while (bi < B && n[bi] == 0) ++bi;
        const int sb = bi, sp = p;
        const int first = bi < B ? count[bi] : 0;
        long long left = budget;
        while (bi < B) {
          const int nb = n[bi];
          if (nb == 0) {
            ++bi;
            continue;
          }
          const int rest = nb - p;
          if (u == U - 1 || rest + kSchedFixedCost <= left) {
            left -= rest + kSchedFixedCost;
            count[bi] += 1;
            ++bi;
            p = 0;
            continue;
          }
          const long long take = left - kSchedFixedCost;
          if (take >= 1) {
            p += static_cast<int>(take);
            count[bi] += 1;
          }
          break;
        }
        put_row(sched + 8 * u, sb, sp, bi, p, first);
      }
    }
    int run = 0;
    num_splits[0] = 0;
    for (int i = 0; i < B; ++i) {
      run += count[i];
      num_splits[i + 1] = run;
    }
  }
}

// Partial slots are [slot][slot_rows] rows of dv = 512; with uniform_splits > 0
// sequence bi owns slots [bi * uniform_splits, (bi + 1) * uniform_splits).
__global__ void split_combine_kernel(const int32_t* __restrict__ num_splits, int uniform_splits,
                                     const float* __restrict__ ws_o, const float2* __restrict__ ws_ml,
                                     const float* __restrict__ ws_d, const float* __restrict__ ws_corr, int apply_corr,
                                     float softmax_scale, uint16_t* __restrict__ out, float* __restrict__ lse, int rows,
                                     int slot_rows) {
  const int bi = blockIdx.x;
  const int r0 = blockIdx.y * 16;
  const int s0 = uniform_splits > 0 ? bi * uniform_splits : num_splits[bi];
  const int ns = uniform_splits > 0 ? uniform_splits : num_splits[bi + 1] - s0;
  if (ns == 1) {
    const int r = r0 + threadIdx.x;
    if (!apply_corr || threadIdx.x >= 16 || r >= rows) return;
    const size_t row = static_cast<size_t>(bi) * rows + r;
    const float l = lse[row];
    if (l != kNegInf) lse[row] = l + ws_corr[2 * row] + ws_corr[2 * row + 1];
    return;
  }
  const int lane = threadIdx.x % 32;
  for (int r = r0 + threadIdx.x / 32; r < min(r0 + 16, rows); r += 4) {
    const size_t row = static_cast<size_t>(bi) * rows + r;
    uint16_t* orow = out + row * kMlaDV + lane * 16;
    float big_m = kNegInf;
    for (int s = 0; s < ns; ++s) big_m = fmaxf(big_m, ws_ml[static_cast<size_t>(s0 + s) * slot_rows + r].x);
    if (ns == 0 || big_m == kNegInf) {  // no visible key: out 0, lse -inf
      *reinterpret_cast<uint4*>(orow) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(orow + 8) = make_uint4(0, 0, 0, 0);
      if (lane == 0) lse[row] = kNegInf;
      continue;
    }
    float acc[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = 0.f;
    float big_l = 0.f, dq = 0.f;
    for (int s = 0; s < ns; ++s) {
      const size_t slot = static_cast<size_t>(s0 + s) * slot_rows + r;
      const float2 ml = ws_ml[slot];
      if (ml.x == kNegInf) continue;  // empty shard: the neutral element
      const float w = ex2_approx(ml.x - big_m);
      big_l += ml.y * w;
      if (apply_corr) dq += w * (ws_d[2 * slot] + ws_d[2 * slot + 1]);
      const float4* src = reinterpret_cast<const float4*>(ws_o + slot * kMlaDV + lane * 16);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 v = src[c];
        acc[4 * c + 0] += w * v.x;
        acc[4 * c + 1] += w * v.y;
        acc[4 * c + 2] += w * v.z;
        acc[4 * c + 3] += w * v.w;
      }
    }
    const float inv = big_l > 0.f ? 1.f / big_l : 0.f;
    uint4 w0, w1;
    w0.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    w0.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    w0.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    w0.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    w1.x = pack_bf16x2(acc[8] * inv, acc[9] * inv);
    w1.y = pack_bf16x2(acc[10] * inv, acc[11] * inv);
    w1.z = pack_bf16x2(acc[12] * inv, acc[13] * inv);
    w1.w = pack_bf16x2(acc[14] * inv, acc[15] * inv);
    *reinterpret_cast<uint4*>(orow) = w0;
    *reinterpret_cast<uint4*>(orow + 8) = w1;
    if (lane == 0)
      lse[row] = big_l > 0.f ? (big_m + lg2_approx(big_l)) * kLn2 - softmax_scale * dq * inv : kNegInf;
  }
}

}  // namespace

cudaError_t launch_mla_metadata(const int32_t* seqlens, int b, int num_units, int force_splits, int32_t* tile_sched,
                                int32_t* num_splits, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(b) * 2 * sizeof(int32_t);
  if (smem > kMetadataMaxSmem) return cudaErrorInvalidValue;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(mla_metadata_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMetadataMaxSmem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  mla_metadata_kernel<<<1, 32, smem, stream>>>(seqlens, b, num_units, force_splits, tile_sched, num_splits);
  return cudaGetLastError();
}

cudaError_t launch_split_combine(const int32_t* num_splits, int uniform_splits, const float* ws_o, const float2* ws_ml,
                                 const float* ws_d, const float* ws_corr, int apply_corr, float softmax_scale,
                                 uint16_t* out, float* lse, int b, int rows, int slot_rows, cudaStream_t stream) {
  if (b == 0) return cudaSuccess;
  dim3 grid(b, (rows + 15) / 16);
  split_combine_kernel<<<grid, 128, 0, stream>>>(num_splits, uniform_splits, ws_o, ws_ml, ws_d, ws_corr, apply_corr,
                                                 softmax_scale, out, lse, rows, slot_rows);
  return cudaGetLastError();
}

cudaError_t launch_mla_combine(const int32_t* num_splits, const float* ws_o, const float2* ws_ml, const float* ws_d,
                               const float* ws_corr, int apply_corr, float softmax_scale, uint16_t* out, float* lse,
                               int b, int rows, cudaStream_t stream) {
  return launch_split_combine(num_splits, 0, ws_o, ws_ml, ws_d, ws_corr, apply_corr, softmax_scale, out, lse, b, rows,
                              kMlaRows, stream);
}

uint32_t metadata_read_and_clear_status() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_meta, sizeof(v));
  cudaMemcpyToSymbol(g_status_meta, &z, sizeof(z));
  return v;
}

}  // namespace fp8mla
