// Tile scheduling for the dense MLA kernel and the split-KV combine kernel.
//
// Scheduling: every non-empty sequence occupies pages + kSchedFixedCost units
// of one cost line (the fixed part stands for its Q load and epilogue); unit
// u takes the cost interval [floor(u W / U), floor((u + 1) W / U)), and a
// cost position maps to a page of its sequence (its first kSchedFixedCost
// positions to page 0).  Units whose interval holds no page are empty.  A
// sequence cut across units becomes several splits whose partial
// (m, l, acc) the combine kernel merges: the split-KV flash-decoding of the
// InfiniCore "FP8(E4M3) KV cache support in paged attention" page (split-kv
// commit), with a balanced persistent schedule instead of a fixed split
// count.  Every step is a prefix sum or an independent binary search.
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

constexpr int kMetaThreads = 512;

// Exclusive prefix sum of v[0, n) in place (one block); returns the total.
// Each thread sums a contiguous run, the runs are scanned with warp shuffles
// (in-warp, then across the warp totals), and each thread rewrites its run.
// scratch holds at least blockDim.x / 32 + 1 values.
template <typename T>
__device__ T block_exclusive_scan(T* v, int n, T* scratch) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, wid = tid >> 5, nw = nt >> 5;
  const int per = (n + nt - 1) / nt;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  T run = 0;
  for (int i = lo; i < hi; ++i) run += v[i];
  T inc = run;  // inclusive scan of the runs inside the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) scratch[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    T w = lane < nw ? scratch[lane] : T(0);
    T winc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += y;
    }
    if (lane < nw) scratch[lane] = winc - w;  // exclusive offset of warp `lane`
    if (lane == 31) scratch[nw] = winc;       // the total
  }
  __syncthreads();
  T acc = scratch[wid] + inc - run;
  for (int i = lo; i < hi; ++i) {
    const T x = v[i];
    v[i] = acc;
    acc += x;
  }
  const T total = scratch[nw];
  __syncthreads();
  return total;
}

// Flattened (sequence, page) position of cost-line position x.
__device__ __forceinline__ void cost_position(const long long* cost0, const int32_t* n, int B, long long x, int& b,
                                              int& p) {
  int lo = 0, hi = B;  // largest b with cost0[b] <= x among non-empty sequences; B if none
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (cost0[mid] <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  b = lo;
  while (b < B && n[b] == 0) ++b;  // cost0 is flat across empty sequences
  if (b >= B) {
    b = B;
    p = 0;
    return;
  }
  const long long off = x - cost0[b] - kSchedFixedCost;
  p = off > 0 ? static_cast<int>(off) : 0;
}

__global__ void __launch_bounds__(kMetaThreads) mla_metadata_kernel(const int32_t* __restrict__ seqlens, int B, int U,
                                                                    int force, int32_t* __restrict__ sched,
                                                                    int32_t* __restrict__ num_splits) {
  extern __shared__ __align__(16) uint8_t meta_raw[];
  long long* cost0 = reinterpret_cast<long long*>(meta_raw);           // [B + 1]
  long long* lscratch = cost0 + (B + 1);                               // [kMetaThreads + 1]
  int32_t* n = reinterpret_cast<int32_t*>(lscratch + kMetaThreads + 1);  // [B]
  int32_t* count = n + B;                                              // [B + 1]
  int32_t* ustart = count + (B + 1);                                   // [2 (U + 1)]
  int32_t* iscratch = ustart + 2 * (U + 1);                            // [kMetaThreads + 1]
  if (blockIdx.x != 0) return;
  griddep_launch_dependents();  // the decode kernel's prologue may overlap this one
  // Launched as a programmatic dependent of whatever the caller enqueued
  // before (which may have written seqlens): wait for it before reading.
  griddep_wait();
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int i = tid; i < B; i += nt) {
    n[i] = pages_of(seqlens[i]);
    count[i] = 0;
  }
  __syncthreads();

  if (force > 0) {
    // chunk j of sequence i (c = min(force, n_i) chunks) goes to unit (number of chunks before i) + j
    for (int i = tid; i < B; i += nt) count[i] = min(force, n[i]);
    __syncthreads();
    block_exclusive_scan<int32_t>(count, B, iscratch);  // count[i] = first unit of sequence i
    for (int i = tid; i < B; i += nt) {
      const int nb = n[i], c = min(force, nb), u0 = count[i];
      for (int j = 0; j < c; ++j) {
        const int u = u0 + j;
        if (u >= U) break;  // the host refuses b * force > num_units
        const int p0 = static_cast<int>((static_cast<long long>(j) * nb) / c);
        const int p1 = static_cast<int>((static_cast<long long>(j + 1) * nb) / c);
        if (p1 == nb)
          put_row(sched + 8 * u, i, p0, i + 1, 0, j);
        else
          put_row(sched + 8 * u, i, p0, i, p1, j);
      }
    }
    const int used = B > 0 ? min(U, count[B - 1] + min(force, n[B - 1])) : 0;
    for (int u = used + tid; u < U; u += nt) put_row(sched + 8 * u, B, 0, B, 0, 0);
    __syncthreads();
    for (int i = tid; i < B; i += nt) count[i] = min(force, n[i]);
  } else {
    for (int i = tid; i < B; i += nt) cost0[i] = n[i] > 0 ? n[i] + kSchedFixedCost : 0;
    __syncthreads();
    const long long W = block_exclusive_scan<long long>(cost0, B, lscratch);
    if (tid == 0) cost0[B] = W;
    __syncthreads();
    // start position of every unit, and of the end (unit U)
    for (int u = tid; u <= U; u += nt) {
      int b, p;
      if (u == U) {
        b = B;
        p = 0;
      } else {
        cost_position(cost0, n, B, (static_cast<long long>(u) * W) / U, b, p);
      }
      ustart[2 * u] = b;
      ustart[2 * u + 1] = p;
    }
    __syncthreads();
    for (int u = tid; u < U; u += nt) {
      const int bs = ustart[2 * u], ps = ustart[2 * u + 1];
      const int be = ustart[2 * u + 2], pe = ustart[2 * u + 3];
      const bool nonempty = (bs < be) || (bs == be && ps < pe);
      // piece index inside sequence bs: piece 0 starts at page 0, and every
      // non-empty unit starting inside it at page > 0 opens the next one
      int first = 0;
      if (nonempty && ps > 0)
        for (int v = u; v >= 0 && ustart[2 * v] == bs; --v) {
          const int vb = ustart[2 * v], vp = ustart[2 * v + 1];
          const bool vne = (vb < ustart[2 * v + 2]) || (vb == ustart[2 * v + 2] && vp < ustart[2 * v + 3]);
          if (vne && vp > 0) ++first;
        }
      put_row(sched + 8 * u, bs, ps, be, pe, first);
      if (nonempty)
        for (int i = bs; i <= min(be, B - 1); ++i) {
          const int lo = (i == bs) ? ps : 0;
          const int hi = (i == be) ? pe : n[i];
          if (hi > lo) atomicAdd(&count[i], 1);
        }
    }
  }
  __syncthreads();
  const int total = block_exclusive_scan<int32_t>(count, B, iscratch);
  for (int i = tid; i < B; i += nt) num_splits[i] = count[i];
  if (tid == 0) num_splits[B] = total;
}

// Grid (sequence, 8-row block), one warp per row, lane j owning dv columns
// [16 j, 16 j + 16).  A sequence with exactly one split was finished by the
// decode kernel: only its LSE correction is left.  Otherwise up to four splits
// are merged with every load issued before any is used, more 32 at a time with
// a rescale of what is accumulated so far between rounds:
// M = max m_s, L = sum l_s 2^(m_s - M), out = sum acc_s 2^(m_s - M) / L,
// lse = ln2 (M + log2 L).  Partial slots are [slot][128] rows of dv = 512
// bf16, sequence bi owning the slots from num_splits[bi].  With q non-null
// every row's LSE also gets the first-order Q-quantisation correction
// lse -= softmax_scale (q_hat - q) . out, from the finished output row and
// q_hat - q of the row's latent part, with the row's power-of-two scale qs
// and the decode kernel's rounding (exact in fp32): q_hat = E4M3(q / qs) qs
// for FP8 dots, q_hat = (hi + E4M3(q / qs - hi)) qs with hi = E4M3(q / qs)
// for two-term dots (two_term != 0).
// (At most 64 registers, four CTAs per SM: its 1 024 CTAs of the b = 64 MTP
// batch then run in fewer waves after the decode kernel; step 65.7 -> 65.4 us
// despite a 48-byte spill.)
__global__ void __launch_bounds__(256, 4) mla_combine_kernel(
    const int32_t* __restrict__ num_splits, const uint16_t* __restrict__ ws_o, const float2* __restrict__ ws_ml,
    const uint16_t* __restrict__ q, const float* __restrict__ qscale, int two_term, float softmax_scale,
    uint16_t* __restrict__ out, float* __restrict__ lse, int rows) {
  const int bi = blockIdx.x;
  const int r = blockIdx.y * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // The split counts and the row scales were final before the decode kernel
  // started (it waited for them), so they are read before waiting for it.
  const int s0 = __ldg(num_splits + bi);
  const int ns = __ldg(num_splits + bi + 1) - s0;
  float ev[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) ev[k] = 0.f;
  if (q != nullptr && r < rows) {
    const size_t row_q = static_cast<size_t>(bi) * rows + r;
    const uint4* qv = reinterpret_cast<const uint4*>(q + row_q * kMlaD) + lane * 2;  // latent dims [16 lane, +16)
    const uint4 a = __ldg(qv), c = __ldg(qv + 1);
    const float qs = __ldg(qscale + static_cast<size_t>(bi) * kMlaRows + r);
    // 1 / qs as the prep kernel forms it: the power of two with the opposite exponent
    const int qe = static_cast<int>((__float_as_uint(qs) >> 23) & 0xFFu) - 127;
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - qe) << 23);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      uint32_t hi, lo;
      split_e4m3x4(bf16_lo(w[k]) * inv, bf16_hi(w[k]) * inv, bf16_lo(w[k + 1]) * inv, bf16_hi(w[k + 1]) * inv, hi,
                   lo);
      if (!two_term) lo = 0u;  // E4M3 zero codes
      const uint32_t h01 = e4m3x2_to_f16x2(hi & 0xFFFFu), h23 = e4m3x2_to_f16x2(hi >> 16);
      const uint32_t l01 = e4m3x2_to_f16x2(lo & 0xFFFFu), l23 = e4m3x2_to_f16x2(lo >> 16);
      ev[2 * k] = (f16_lo(h01) + f16_lo(l01)) * qs - bf16_lo(w[k]);
      ev[2 * k + 1] = (f16_hi(h01) + f16_hi(l01)) * qs - bf16_hi(w[k]);
      ev[2 * k + 2] = (f16_lo(h23) + f16_lo(l23)) * qs - bf16_lo(w[k + 1]);
      ev[2 * k + 3] = (f16_hi(h23) + f16_hi(l23)) * qs - bf16_hi(w[k + 1]);
    }
  }
  // (q_hat - q) . o over the whole row, o holding this lane's 16 columns
  auto err_dot = [&](const float (&o)[16]) {
    float d = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) d += ev[2 * k] * o[2 * k] + ev[2 * k + 1] * o[2 * k + 1];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    return d;
  };
  // (no early trigger for the caller's next kernel: a dependent launched early, such as
  // the next step's scheduler and Q prep, holds SM resources this grid's later CTAs need;
  // the dense MLA step measured 65.5 us without it, 66.0 with)
  griddep_wait();  // launched as a dependent of the decode kernel
  if (r >= rows) return;
  const size_t row = static_cast<size_t>(bi) * rows + r;
  uint16_t* orow = out + row * kMlaDV + lane * 16;
  if (ns == 1) {
    if (q != nullptr) {
      const uint4 a = reinterpret_cast<const uint4*>(orow)[0], b2 = reinterpret_cast<const uint4*>(orow)[1];
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w};
      float o[16];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        o[2 * q] = bf16_lo(w[q]);
        o[2 * q + 1] = bf16_hi(w[q]);
      }
      const float d = err_dot(o);
      if (lane == 0) {
        const float l = lse[row];
        if (l != kNegInf) lse[row] = l - softmax_scale * d;
      }
    }
    return;
  }
  if (ns <= 0) {
    *reinterpret_cast<uint4*>(orow) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(orow + 8) = make_uint4(0, 0, 0, 0);
    if (lane == 0) lse[row] = kNegInf;
    return;
  }
  float acc[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) acc[c] = 0.f;
  float big_l = 0.f, big_m = kNegInf;
  // acc += wj * (this lane's 16 columns of split j's partial row)
  auto load_partial = [&](int j, uint4 (&v)[2]) {
    const size_t slot = static_cast<size_t>(s0 + j) * kMlaRows + r;
    const uint4* src = reinterpret_cast<const uint4*>(ws_o + slot * kMlaDV + lane * 16);
    v[0] = __ldg(src);
    v[1] = __ldg(src + 1);
  };
  auto accumulate = [&](float wj, const uint4 (&v)[2]) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[8 * c + 2 * q] += wj * bf16_lo(w4[q]);
        acc[8 * c + 2 * q + 1] += wj * bf16_hi(w4[q]);
      }
    }
  };
  if (ns <= 4) {
    // few splits (the usual case): every load is issued before any is used
    constexpr int kMax = 4;
    uint4 v[kMax][2];
#pragma unroll
    for (int j = 0; j < kMax; ++j)
      if (j < ns) load_partial(j, v[j]);
    const float2 ml =
        lane < ns ? __ldg(ws_ml + static_cast<size_t>(s0 + lane) * kMlaRows + r) : make_float2(kNegInf, 0.f);
    float m_all = ml.x;
#pragma unroll
    for (int o = 2; o > 0; o >>= 1) m_all = fmaxf(m_all, __shfl_xor_sync(0xffffffffu, m_all, o));
    m_all = __shfl_sync(0xffffffffu, m_all, 0);
    if (m_all != kNegInf) {
      big_m = m_all;
      const float w = (ml.x == kNegInf) ? 0.f : ex2_approx(ml.x - big_m);  // an empty split adds nothing
      big_l = ml.y * w;
#pragma unroll
      for (int j = 0; j < kMax; ++j)
        if (j < ns) accumulate(__shfl_sync(0xffffffffu, w, j), v[j]);
    }
  } else {
    for (int base = 0; base < ns; base += 32) {
      // this round's splits: lane j holds split base + j's (m, l)
      const int cnt = min(32, ns - base);
      const float2 ml = lane < cnt ? __ldg(ws_ml + static_cast<size_t>(s0 + base + lane) * kMlaRows + r)
                                   : make_float2(kNegInf, 0.f);
      float m_round = ml.x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m_round = fmaxf(m_round, __shfl_xor_sync(0xffffffffu, m_round, o));
      if (m_round == kNegInf) continue;  // every split of this round is empty
      // fold this round into the running (big_m, big_l, acc)
      const float m_new = fmaxf(big_m, m_round);
      const float a_old = (big_m == kNegInf) ? 0.f : ex2_approx(big_m - m_new);
      big_l *= a_old;
#pragma unroll
      for (int c = 0; c < 16; ++c) acc[c] *= a_old;
      big_m = m_new;
      const float w = (ml.x == kNegInf) ? 0.f : ex2_approx(ml.x - big_m);  // an empty split is the neutral element
      big_l += ml.y * w;
#pragma unroll 4
      for (int j = 0; j < cnt; ++j) {
        uint4 v[2];
        load_partial(base + j, v);
        accumulate(__shfl_sync(0xffffffffu, w, j), v);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) big_l += __shfl_xor_sync(0xffffffffu, big_l, o);
  const float inv = big_l > 0.f ? 1.f / big_l : 0.f;
#pragma unroll
  for (int c = 0; c < 16; ++c) acc[c] *= inv;
  const float d = q != nullptr ? err_dot(acc) : 0.f;  // the LSE correction from the merged output row
  uint4 w0, w1;
  w0.x = pack_bf16x2(acc[0], acc[1]);
  w0.y = pack_bf16x2(acc[2], acc[3]);
  w0.z = pack_bf16x2(acc[4], acc[5]);
  w0.w = pack_bf16x2(acc[6], acc[7]);
  w1.x = pack_bf16x2(acc[8], acc[9]);
  w1.y = pack_bf16x2(acc[10], acc[11]);
  w1.z = pack_bf16x2(acc[12], acc[13]);
  w1.w = pack_bf16x2(acc[14], acc[15]);
  *reinterpret_cast<uint4*>(orow) = w0;
  *reinterpret_cast<uint4*>(orow + 8) = w1;
  if (lane == 0) lse[row] = big_l > 0.f ? (big_m + lg2_approx(big_l)) * kLn2 - softmax_scale * d : kNegInf;
}

}  // namespace

size_t metadata_smem_bytes(int b, int num_units) {
  return static_cast<size_t>(b + 1 + kMetaThreads + 1) * sizeof(long long) +
         static_cast<size_t>(b + (b + 1) + 2 * (num_units + 1) + kMetaThreads + 1) * sizeof(int32_t);
}

cudaError_t launch_mla_metadata(const int32_t* seqlens, int b, int num_units, int force_splits, int32_t* tile_sched,
                                int32_t* num_splits, cudaStream_t stream) {
  const size_t smem = metadata_smem_bytes(b, num_units);
  if (smem > kMetadataMaxSmem) return cudaErrorInvalidValue;
  static std::atomic<uint64_t> configured{0};  // per device: CUDA keeps the limit per device
  const cudaError_t e = configure_once(configured, [] {
    return cudaFuncSetAttribute(mla_metadata_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kMetadataMaxSmem));
  });
  if (e != cudaSuccess) return e;
  // a programmatic dependent: its launch overlaps the tail of the previous kernel
  return launch_dependent(mla_metadata_kernel, dim3(1), dim3(kMetaThreads), smem, stream, seqlens, b, num_units,
                          force_splits, tile_sched, num_splits);
}

cudaError_t launch_mla_combine(const int32_t* num_splits, const uint16_t* ws_o, const float2* ws_ml,
                               const uint16_t* q, const float* qscale, bool two_term, float softmax_scale,
                               uint16_t* out, float* lse, int b, int rows, cudaStream_t stream) {
  if (b == 0) return cudaSuccess;
  return launch_dependent(mla_combine_kernel, dim3(b, (rows + 7) / 8), dim3(256), 0, stream, num_splits, ws_o, ws_ml,
                          q, qscale, two_term ? 1 : 0, softmax_scale, out, lse, rows);
}

uint32_t metadata_read_and_clear_status() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_meta, sizeof(v));
  cudaMemcpyToSymbol(g_status_meta, &z, sizeof(z));
  return v;
}

}  // namespace fp8mla
