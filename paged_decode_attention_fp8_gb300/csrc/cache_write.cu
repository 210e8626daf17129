// FP8 (E4M3) paged KV-cache write: quantise new K or V rows on their way into
// the cache.
//
// InfiniCore "add FP8 blockwise dequantize/GEMM operators and FP8(E4M3) KV
// cache support in paged attention", Summary (paged_caching): a write kernel
// over (token, kv_head) rows reduces each row's amax, stores the row's scale
// amax / 448 (1 for an all-zero row) in a [num_blocks, h_kv, page] float32
// array, and encodes the row as E4M3.  The same kernel also writes with one
// given per-tensor scale, the form the dense MLA and GQA decode kernels read.
//
// Per row: scale = fp32(amax / 448) (1 for an all-zero row) is what the
// cache keeps; the codes use its reciprocal inv = fp32(448 / amax) (1 for a
// zero row), one IEEE division per row: code = E4M3(fp32(x * inv)), rounded
// to nearest even and saturated to +-448.  A row with amax < 2^-64 is first
// lifted by 2^64 (exact: a power of two, and no such row can overflow), so
// inv never overflows.  Per-tensor mode: inv = fp32(1 / scale).
// Token t's row for head h lands in slot s = slot_mapping[t]
// (block s / page, offset s % page); a negative slot skips the token, a slot
// past the cache sets FP8MLA_DEV_BAD_SLOT and skips it.
//
// HBM-bound streaming.  A group of L lanes owns a row: the fewest (a power of
// two, at most 32) that leave each lane at most three of the row's 16-byte
// chunks, so a lane holds two chunks of a power-of-two row and the row's
// index arithmetic, done by every lane of the group, is spread over 32 bytes
// or more.  Each warp walks its rows in a grid-stride loop (four CTAs per SM),
// R rows per group per step (R = 2 when a lane holds one or two chunks of a
// row, else 1), with the next step's 16-byte loads issued before the current
// step is worked on.  A step reduces each row's amax across its group with shuffles;
// lane r of the group divides for row r and hands the reciprocal round by
// shuffle (and stores row r's scale), so a lane does one division per step;
// then each lane stores 8 codes per chunk.  Integer division by h_kv and the
// page size uses a multiply-high by a precomputed constant (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994),
// exact for numerators below 2^31.
#include <cuda_runtime.h>

#include <cstdint>

#include "cache_write.h"
#include "common.cuh"

namespace fp8mla {
namespace {

__device__ uint32_t g_status_cw;

constexpr int kCwThreads = 256;

// n / d by a multiply-high (see make_fast_div)
struct FastDiv {
  uint32_t d, m, s;
};
constexpr int kCwMaxChunks = 4;  // 16-byte chunks (8 bf16) a lane holds per row; head_dim <= 8 * 32 * 4

constexpr float kTinyAmax = 5.42101086242752217e-20f;  // 2^-64
constexpr float kTinyLift = 1.84467440737095516e19f;   // 2^64

// |x| of a bf16 pair's two halves, max with m
__device__ __forceinline__ float absmax_bf16x2(float m, uint32_t w) {
  return fmax3(m, __uint_as_float((w & 0x7FFFu) << 16), __uint_as_float(w & 0x7FFF0000u));
}

// Two bf16 halves times inv, then E4M3 (low half in the low byte).
__device__ __forceinline__ uint32_t encode_bf16x2(uint32_t w, float inv) {
  return pack_e4m3x2(__fmul_rn(bf16_lo(w), inv), __fmul_rn(bf16_hi(w), inv));
}

// The same for a lifted row: times 2^64 first (exact), then times inv.
__device__ __forceinline__ uint32_t encode_bf16x2_lifted(uint32_t w, float inv) {
  return pack_e4m3x2(__fmul_rn(__fmul_rn(bf16_lo(w), kTinyLift), inv),
                     __fmul_rn(__fmul_rn(bf16_hi(w), kTinyLift), inv));
}

__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
  return f.d == 1 ? n : (__umulhi(n, f.m) >> f.s);
}

// Rows per group per step: two while a lane holds at most two chunks of a
// row (four 16-byte loads in flight per lane), else one.
template <int kC>
__host__ __device__ constexpr int rows_per_step() {
  return kC >= 3 ? 1 : 2;
}

template <int kR, int kC>
struct CwStep {
  uint4 v[kR][kC];
  int32_t slot[kR];
};

template <int kL, int kC>
__global__ void __launch_bounds__(kCwThreads, 4) cache_write_kernel(
    const uint16_t* __restrict__ x, int64_t x_token_stride, const int32_t* __restrict__ slot_mapping,
    uint32_t n_rows, FastDiv div_h, int head_dim, FastDiv div_page, uint32_t num_slots, uint8_t* __restrict__ cache,
    const float* __restrict__ tensor_scale, float* __restrict__ token_scales) {
  constexpr int kR = rows_per_step<kC>();
  constexpr int kWarpRows = (32 / kL) * kR;  // rows a warp takes per step
  constexpr bool kSpread = kL >= kR;         // a group has a lane for each of its rows' divisions
  const int lane = threadIdx.x % 32;
  const int sub = lane % kL;                 // this lane's place in its row's group
  const int grp = lane / kL;
  const uint32_t warp_id = blockIdx.x * (kCwThreads / 32) + threadIdx.x / 32;
  const uint32_t stride = gridDim.x * (kCwThreads / 32) * kWarpRows;
  const uint32_t h_kv = div_h.d;
  const uint32_t page = div_page.d;
  const int chunks = head_dim / 8;
  const bool per_row = token_scales != nullptr;
  const float tensor_inv = per_row ? 1.f : __fdiv_rn(1.f, __ldg(tensor_scale));

  auto load = [&](uint32_t base, CwStep<kR, kC>& st) {
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      const uint32_t row = base + grp * kR + r;
      st.slot[r] = -1;
#pragma unroll
      for (int i = 0; i < kC; ++i) st.v[r][i] = make_uint4(0, 0, 0, 0);
      if (row < n_rows) {
        const uint32_t token = fast_div(row, div_h);
        const uint32_t head = row - token * h_kv;
        st.slot[r] = __ldg(slot_mapping + token);
        const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(token) * x_token_stride +
                                                          static_cast<int64_t>(head) * head_dim);
#pragma unroll
        for (int i = 0; i < kC; ++i) {
          const int c = sub + i * kL;
          if (c < chunks) st.v[r][i] = __ldcs(src + c);
        }
      }
    }
  };

  auto process = [&](uint32_t base, const CwStep<kR, kC>& st) {
    float amax[kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      amax[r] = 0.f;
#pragma unroll
      for (int i = 0; i < kC; ++i) {
        amax[r] = absmax_bf16x2(amax[r], st.v[r][i].x);
        amax[r] = absmax_bf16x2(amax[r], st.v[r][i].y);
        amax[r] = absmax_bf16x2(amax[r], st.v[r][i].z);
        amax[r] = absmax_bf16x2(amax[r], st.v[r][i].w);
      }
#pragma unroll
      for (int off = kL / 2; off > 0; off >>= 1)
        amax[r] = fmaxf(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], off));
    }
    float inv[kR];
    float my_scale = 1.f;  // kSpread: the scale of row `sub` of this group
    if (per_row) {
      if constexpr (kSpread) {
        float a = amax[0];
#pragma unroll
        for (int r = 1; r < kR; ++r)
          if (sub == r) a = amax[r];
        const float mine = a > 0.f ? __fdiv_rn(448.f, a < kTinyAmax ? __fmul_rn(a, kTinyLift) : a) : 1.f;
        my_scale = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
#pragma unroll
        for (int r = 0; r < kR; ++r) inv[r] = __shfl_sync(0xffffffffu, mine, (lane & ~(kL - 1)) + r);
      } else {
#pragma unroll
        for (int r = 0; r < kR; ++r)
          inv[r] = amax[r] > 0.f ? __fdiv_rn(448.f, amax[r] < kTinyAmax ? __fmul_rn(amax[r], kTinyLift) : amax[r])
                                 : 1.f;
      }
    } else {
#pragma unroll
      for (int r = 0; r < kR; ++r) inv[r] = tensor_inv;
    }
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      const int32_t slot = st.slot[r];
      if (slot < 0) continue;  // padding, or past the last row
      if (static_cast<uint32_t>(slot) >= num_slots) {
        if (sub == 0) atomicOr(&g_status_cw, FP8MLA_DEV_BAD_SLOT);
        continue;
      }
      const uint32_t row = base + grp * kR + r;
      const uint32_t head = row - fast_div(row, div_h) * h_kv;
      const uint32_t block = fast_div(static_cast<uint32_t>(slot), div_page);
      const int64_t dst_row = (static_cast<int64_t>(block) * h_kv + head) * page + (slot - block * page);
      uint2* dst = reinterpret_cast<uint2*>(cache + dst_row * head_dim);
      const bool lifted = per_row && amax[r] < kTinyAmax;
#pragma unroll
      for (int i = 0; i < kC; ++i) {
        const int c = sub + i * kL;
        if (c < chunks) {
          uint2 o;
          if (!lifted) {
            o.x = encode_bf16x2(st.v[r][i].x, inv[r]) | (encode_bf16x2(st.v[r][i].y, inv[r]) << 16);
            o.y = encode_bf16x2(st.v[r][i].z, inv[r]) | (encode_bf16x2(st.v[r][i].w, inv[r]) << 16);
          } else {
            o.x = encode_bf16x2_lifted(st.v[r][i].x, inv[r]) | (encode_bf16x2_lifted(st.v[r][i].y, inv[r]) << 16);
            o.y = encode_bf16x2_lifted(st.v[r][i].z, inv[r]) | (encode_bf16x2_lifted(st.v[r][i].w, inv[r]) << 16);
          }
          dst[c] = o;
        }
      }
      if (per_row) {
        if constexpr (kSpread) {
          if (sub == r) token_scales[dst_row] = my_scale;
        } else {
          if (sub == 0) token_scales[dst_row] = amax[r] > 0.f ? __fdiv_rn(amax[r], 448.f) : 1.f;
        }
      }
    }
  };

  // two steps in flight per warp: the next step's loads go out before this one is worked on
  uint32_t base = warp_id * kWarpRows;
  if (base >= n_rows) return;  // the same for the whole warp
  CwStep<kR, kC> a, b;
  load(base, a);
  for (;;) {
    const uint32_t nb = base + stride;  // < 2^32: both terms are below 2^31
    const bool more = nb < n_rows;
    if (more) load(nb, b);
    process(base, a);
    if (!more) break;
    base = nb;
    const uint32_t nb2 = base + stride;
    const bool more2 = nb2 < n_rows;
    if (more2) load(nb2, a);
    process(base, b);
    if (!more2) break;
    base = nb2;
  }
}

// Constants of fast_div for divisor d (numerators below 2^31): with
// l = ceil(log2 d), m = floor(2^(31 + l) / d) + 1 < 2^32 gives
// n / d = (n * m) >> (31 + l) for every n < 2^31 (d = 1 is passed through).
FastDiv make_fast_div(int d) {
  FastDiv f;
  f.d = static_cast<uint32_t>(d);
  f.m = 0;
  f.s = 0;
  if (d <= 1) return f;
  uint32_t l = 0;
  while ((1ull << l) < static_cast<uint64_t>(d)) ++l;
  f.m = static_cast<uint32_t>((1ull << (31 + l)) / static_cast<uint64_t>(d) + 1);
  f.s = l - 1;
  return f;
}

// SM count of the current device, queried once per device (152 if unknown).
int device_sms() {
  static std::atomic<int> sms[64];  // zero-initialised: static storage
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  int n = sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 152;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <int kL, int kC>
cudaError_t launch_cw(const CacheWriteArgs& a, cudaStream_t stream) {
  constexpr int kBlockRows = (kCwThreads / 32) * (32 / kL) * rows_per_step<kC>();
  const int64_t rows = static_cast<int64_t>(a.n_tokens) * a.h_kv;
  const int64_t need = (rows + kBlockRows - 1) / kBlockRows;
  const int64_t cap = static_cast<int64_t>(device_sms()) * 4;  // one wave of resident CTAs
  const int64_t blocks = need < cap ? need : cap;
  cache_write_kernel<kL, kC><<<static_cast<unsigned>(blocks), kCwThreads, 0, stream>>>(
      a.x, a.x_token_stride, a.slot_mapping, static_cast<uint32_t>(rows), make_fast_div(a.h_kv), a.head_dim,
      make_fast_div(a.page_size), static_cast<uint32_t>(static_cast<int64_t>(a.num_blocks) * a.page_size), a.cache,
      a.tensor_scale, a.token_scales);
  return cudaGetLastError();
}

}  // namespace

int cache_write_group_lanes(int head_dim) {
  const int chunks = head_dim / 8;
  int l = 1;
  while (l < 32 && (chunks + l - 1) / l > 3) l *= 2;
  return l;
}

fp8mla_status_t cache_write_entry(const CacheWriteArgs& a, cudaStream_t stream) {
  if (a.n_tokens < 0 || a.h_kv < 1 || a.page_size < 1 || a.num_blocks < 1) return FP8MLA_ERR_INVALID_ARG;
  if (a.head_dim < 8 || a.head_dim % 8 != 0 || a.head_dim > 8 * 32 * kCwMaxChunks) return FP8MLA_ERR_INVALID_ARG;
  if ((a.tensor_scale == nullptr) == (a.token_scales == nullptr)) return FP8MLA_ERR_INVALID_ARG;
  if (a.x_token_stride < static_cast<int64_t>(a.h_kv) * a.head_dim || a.x_token_stride % 8 != 0)
    return FP8MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(a.n_tokens) * a.h_kv >= (1ll << 31) ||
      static_cast<int64_t>(a.num_blocks) * a.page_size >= (1ll << 31))
    return FP8MLA_ERR_INVALID_ARG;
  if (a.n_tokens == 0) return FP8MLA_OK;
  if (a.x == nullptr || a.slot_mapping == nullptr || a.cache == nullptr) return FP8MLA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(a.x) % 16 != 0 || reinterpret_cast<uintptr_t>(a.cache) % 16 != 0 ||
      (a.token_scales != nullptr && reinterpret_cast<uintptr_t>(a.token_scales) % 4 != 0))
    return FP8MLA_ERR_INVALID_ARG;
  const int l = cache_write_group_lanes(a.head_dim);
  const int c = (a.head_dim / 8 + l - 1) / l;  // chunks per lane: <= 3 below 32 lanes, <= 4 at 32
  cudaError_t e;
  switch (l * 8 + c) {
    case 1 * 8 + 1: e = launch_cw<1, 1>(a, stream); break;
    case 1 * 8 + 2: e = launch_cw<1, 2>(a, stream); break;
    case 1 * 8 + 3: e = launch_cw<1, 3>(a, stream); break;
    case 2 * 8 + 2: e = launch_cw<2, 2>(a, stream); break;
    case 2 * 8 + 3: e = launch_cw<2, 3>(a, stream); break;
    case 4 * 8 + 2: e = launch_cw<4, 2>(a, stream); break;
    case 4 * 8 + 3: e = launch_cw<4, 3>(a, stream); break;
    case 8 * 8 + 2: e = launch_cw<8, 2>(a, stream); break;
    case 8 * 8 + 3: e = launch_cw<8, 3>(a, stream); break;
    case 16 * 8 + 2: e = launch_cw<16, 2>(a, stream); break;
    case 16 * 8 + 3: e = launch_cw<16, 3>(a, stream); break;
    case 32 * 8 + 2: e = launch_cw<32, 2>(a, stream); break;
    case 32 * 8 + 3: e = launch_cw<32, 3>(a, stream); break;
    case 32 * 8 + 4: e = launch_cw<32, 4>(a, stream); break;
    default: return FP8MLA_ERR_INVALID_ARG;
  }
  return e == cudaSuccess ? FP8MLA_OK : FP8MLA_ERR_CUDA;
}

uint32_t cache_write_read_and_clear_status() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_cw, sizeof(v));
  cudaMemcpyToSymbol(g_status_cw, &z, sizeof(z));
  return v;
}

}  // namespace fp8mla
