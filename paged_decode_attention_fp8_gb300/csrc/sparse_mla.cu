// Top-k sparse MLA decode, tcgen05 + TMA gather4, sm_103a.
//
// The operation (aiter "Support fp8 KV caches and fp8 dots in
// sparse_mla_fwd on gfx942": Results shape -- 16 heads, rope-free d = dv =
// 512, top-k 2048 of one flat E4M3 cache): for each query token t and head h,
//   out[t, h] = softmax_j(scale * q[t, h] . k_j) @ v_j,  j over topk_idx[t]
// with V = K (the same 512 cached values) and index -1 meaning "no key".
//
// GB300 design (swap-AB, one CTA per (token, split of the key list)):
//   * 128 keys per step, gathered into four 128-byte-swizzled atoms (one per
//     128-byte column box) by two engines at once: 32 rows by TMA
//     tile::gather4 from warp 0 (four rows of one column box per
//     instruction), 96 by 16-byte cp.async from warps 2 and 3 (one warp
//     instruction per row); the next step's indices load while a step
//     issues.  The TMA unit takes ~29 ns per gather4 request (all 128 rows
//     through it: 3.7 us per step), and the cp.async rows are limited by the
//     misses an SM keeps in flight; at s_q = 16384 a 32-row TMA share ran
//     3.56 ms per call against 4.07 ms with no TMA rows and 5.43 ms with 64.
//     Index -1 and out-of-range rows land as zeros (the TMA copy's
//     out-of-bounds fill; cp.async with no source bytes) and are masked by
//     select.
//   * S^T = K Q^T on tcgen05 kind::f8f6f4: M = 128 keys, N = 16 heads,
//     K = 512 (16 MMAs); Q is quantised in-kernel per head with a power-of-
//     two scale (aiter page, Technical details: in-kernel Q quantisation),
//     and its rounding error q_hat - q (exact in bf16) is kept in shared
//     memory for the epilogue's LSE correction.
//     S^T lives in TMEM: thread j of the softmax warpgroup owns key j.
//   * Softmax across TMEM lanes: per-head max by warp shuffles + a 4-warp
//     exchange, lazily raised (threshold 1 in log2 units so 128 p <= 256);
//     each thread keeps its own partial row sums, reduced once at the end.
//   * P is quantised as E4M3(128 p) (aiter page: the x128 scale keeps the
//     softmax tail from flushing to zero; Accuracy: the +9-over-2047 case)
//     and written to shared memory as the K-major B operand.
//   * O^T = V^T P^T in four M = 128 tiles (dv = 512), A = the same gathered
//     atoms read MN-major (no transpose), B = P^T.  O^T sits in TMEM.
//   * Split-KV: shards publish (m, l, acc, (q_hat - q) . acc) and the
//     combine kernel merges them (InfiniCore split-kv commit); with up to 16
//     splits each of its threads loads every split's (m, l, d) with its own
//     partial columns, so the merge is one round trip and has no barrier.
//     (Merging inside a cooperatively launched decode grid was tried: the
//     cooperative launch alone cost ~4.6 us per call at s_q = 2, more than
//     the combine kernel; so was merging inside thread-block clusters over
//     distributed shared memory: slower at s_q = 2 and 16.)  Because V = K, the first-order LSE error of Q's
//     quantisation is scale * (q_hat - q) . out, which the epilogue (or the
//     combine) subtracts.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "mla_decode.h"
#include "sparse_mla.h"

namespace fp8mla {

__device__ uint32_t g_status_sparse;

namespace sparse {

constexpr int kD = 512;
constexpr int kKeys = 128;          // keys per step (MMA M)
constexpr int kN = 16;              // heads (MMA N)
constexpr int kThreads = 256;
constexpr int kStages = 3;
constexpr int kAtom = kKeys * 128;  // one 128-byte column slice of a step (16 KB)
constexpr int kStageBytes = 4 * kAtom;
constexpr int kQBytes = 4 * kN * 128;   // Q tile: 4 atoms x [16 rows x 128 B]
constexpr int kPBytes = kN * 128;       // P^T tile: [16 rows x 128 keys]
constexpr int kEBytes = kN * kD * 2;    // Q's rounding error q_hat - q, bf16 [16 heads][512]
constexpr int kTmaKeys = 32;            // rows of a step gathered by TMA; the rest by cp.async
constexpr int kCopyWarps = 2;           // warps 2 and 3 issue the cp.async rows
constexpr float kPScale = 128.0f;
constexpr float kTau = 1.0f;
constexpr uint32_t kTmemCols = 128;     // S^T 16 + O^T 64
constexpr uint32_t kTS = 0, kTO = 16;

struct Params {
  const uint16_t* q;       // bf16 [s_q, h_q, 512]
  const uint8_t* kv;       // E4M3 [num_tokens, 512]
  const int32_t* idx;      // [s_q, topk]
  const float* kv_scale;
  uint16_t* out;           // bf16 [s_q, h_q, 512]
  float* lse;              // [s_q, h_q]
  float* ws_o;             // [s_q * splits, 16, 512]
  float2* ws_ml;           // [s_q * splits, 16]
  float* ws_d;             // [s_q * splits, 16, 2]
  long long num_tokens;
  float softmax_scale;
  int topk, s_q, h_q, splits, chunks;
};

struct Smem {
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full, s_free, p_full, pv_done, q_full, final_mma, xchg;
  uint32_t tmem_base, abort_flag;
  float qs[kN];
  float red[2][4][kN];   // per-warp partial maxima, double-buffered by step parity
  float red2[4][kN];
};

constexpr size_t kSmemBytes = kStages * kStageBytes + kQBytes + kPBytes + kEBytes + sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "fits the 227 KB opt-in shared memory of a CTA");

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  const bool ok = wait_bounded(bar, parity, abort_flag, &g_status_sparse);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ int pow2_exp_448(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  const int expo = static_cast<int>((bits >> 23) & 0xFFu);
  if (expo == 0) return -126;
  const uint32_t mant = bits & 0x7FFFFFu;
  return max((expo - 127) - (mant <= 0x600000u ? 8 : 7), -126);
}

__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// Is key slot k of token t a real key?  (k past topk, index -1: no; out of range: flagged, no.)
__device__ __forceinline__ int key_row(const Params& p, int t, int k) {
  if (k >= p.topk) return -1;
  const int v = p.idx[static_cast<size_t>(t) * p.topk + k];
  if (v < -1 || v >= p.num_tokens) {
    atomicOr(&g_status_sparse, FP8MLA_DEV_BAD_INDEX);
    return -1;
  }
  return v;
}

// A loaded index as a cache row: -1 (no key) stays -1; out of range is flagged and skipped.
__device__ __forceinline__ int checked_row(const Params& p, int v) {
  if (v < -1 || v >= p.num_tokens) {
    atomicOr(&g_status_sparse, FP8MLA_DEV_BAD_INDEX);
    return -1;
  }
  return v;
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_rows, const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* q_tile = smem + kStages * kStageBytes;
  uint8_t* p_tile = q_tile + kQBytes;
  uint8_t* e_tile = p_tile + kPBytes;
  Smem* sm = reinterpret_cast<Smem*>(e_tile + kEBytes);
  volatile uint32_t* abort_flag = &sm->abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int t = blockIdx.x / prm.splits;       // query token
  const int split = blockIdx.x % prm.splits;
  const int c0 = static_cast<int>((static_cast<long long>(split) * prm.chunks) / prm.splits);
  const int c1 = static_cast<int>((static_cast<long long>(split + 1) * prm.chunks) / prm.splits);
  const int nchunks = c1 - c0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm->kv_full[s], 1 + 32 * kCopyWarps);  // the TMA warp's arrival + one per copying lane
      mbar_init(&sm->kv_empty[s], 1);
    }
    mbar_init(&sm->s_full, 1);
    mbar_init(&sm->s_free, 4);
    mbar_init(&sm->p_full, 4);
    mbar_init(&sm->pv_done, 1);
    mbar_init(&sm->q_full, 4);
    mbar_init(&sm->final_mma, 1);
    mbar_init(&sm->xchg, 4);
    sm->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  griddep_wait();  // inputs may come from the previous kernel in the stream
  // The first step's indices (gather warps) and Q (softmax warps) are loaded
  // before the block-wide barrier, so their latency overlaps it.
  const int32_t* idx_t = prm.idx + static_cast<size_t>(t) * prm.topk;
  auto load_idx = [&](int ch, int (&v)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int k = (c0 + ch) * kKeys + 4 * lane + q;
      v[q] = k < prm.topk ? __ldg(idx_t + k) : -1;
    }
  };
  int raw[4] = {-1, -1, -1, -1};
  if ((warp == 0 || warp == 2 || warp == 3) && nchunks > 0) load_idx(0, raw);
  uint4 qv[8];
  if (warp >= 4) {
    const int qh = (threadIdx.x - 128) / 8, qj = (threadIdx.x - 128) % 8;
    const uint4* qsrc = reinterpret_cast<const uint4*>(prm.q + (static_cast<size_t>(t) * prm.h_q + qh) * kD + qj * 64);
#pragma unroll
    for (int c = 0; c < 8; ++c) qv[c] = qh < prm.h_q ? __ldg(qsrc + c) : make_uint4(0, 0, 0, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = sm->tmem_base;

  if (warp == 0 || warp == 2 || warp == 3) {
    // ------------------------------- gather producers (warps 0, 2, 3) ----
    // Key k of a step (k = 4 j + q) comes from lane j's q-th index.  Rows
    // [0, kTmaKeys): TMA gather4 from warp 0 (four rows of one column box per
    // instruction).  The other rows: cp.async from warps 2 and 3, index lanes
    // in turn; a row is one warp instruction, lane l copying its bytes
    // [16 l, 16 l + 16) into column box l / 8 as 16-byte chunk l % 8,
    // XOR-swizzled by the row (128-byte swizzle).  Each copying lane arrives on
    // the stage's full barrier once its copies land.  The next step's indices
    // are loaded while this step's copies issue.
    const int cw = warp - 2;  // copy warp 0 or 1 (warp 0: the TMA warp)
    const int cb = lane / 8, cc = lane % 8;
    if (warp == 0 && lane == 0) tma_prefetch_desc(&tm_rows);
    int i = 0;
    for (; i < nchunks; ++i) {
      const int st = i % kStages, use = i / kStages;
      int nxt[4] = {-1, -1, -1, -1};
      if (i + 1 < nchunks) load_idx(i + 1, nxt);
      bool ok = true;
      if (lane == 0) ok = use == 0 || wait_bounded(&sm->kv_empty[st], (use - 1) & 1, abort_flag, &g_status_sparse);
      if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) break;
      const int r0 = checked_row(prm, raw[0]), r1 = checked_row(prm, raw[1]);
      const int r2 = checked_row(prm, raw[2]), r3 = checked_row(prm, raw[3]);
      uint8_t* sb = smem + st * kStageBytes;
      if (warp == 0) {
        if (lane == 0) mbar_arrive_expect_tx(&sm->kv_full[st], kTmaKeys * kD);
        __syncwarp();
        if (lane < kTmaKeys / 4) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tma_gather4(sb + j * kAtom + (4 * lane) * 128, &tm_rows, &sm->kv_full[st], j * 128, r0, r1, r2, r3);
        }
      } else {
#pragma unroll 1
        for (int src = kTmaKeys / 4 + cw; src < 32; src += kCopyWarps) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kk = 4 * src + q;
            const int row = __shfl_sync(0xffffffffu, q == 0 ? r0 : (q == 1 ? r1 : (q == 2 ? r2 : r3)), src);
            cp_async16(smem_u32(sb + cb * kAtom + kk * 128 + ((cc ^ (kk & 7)) << 4)),
                       prm.kv + static_cast<size_t>(row >= 0 ? row : 0) * kD + 16 * lane, row >= 0 ? 16u : 0u);
          }
        }
        cp_async_mbar_arrive(&sm->kv_full[st]);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) raw[q] = nxt[q];
    }
    cp_async_wait_all();  // this lane's copies have landed before the CTA can exit
    if (warp == 0 && lane == 0)
      for (int j = max(0, i - kStages); j < i; ++j)
        wait_bounded(&sm->kv_full[j % kStages], (j / kStages) & 1, nullptr, &g_status_sparse);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer ----
    // The whole warp runs the loop (warp-uniform descriptors) and one elected
    // lane issues: from a lone thread each MMA costs about twice as long.
    {
      constexpr uint32_t idesc_qk = make_idesc(0, 0, 0, 0, kN, 128);   // K (K-major) x Q (K-major)
      constexpr uint32_t idesc_pv = make_idesc(0, 0, 1, 0, kN, 128);   // V^T (MN-major) x P^T (K-major)
      const bool leader = elect_one();
      const uint32_t qb = smem_u32(q_tile), pb = smem_u32(p_tile);
      bool ok = warp_wait(&sm->q_full, 0, abort_flag);
      auto issue_pv = [&](int j) -> bool {
        if (!warp_wait(&sm->p_full, j & 1, abort_flag)) return false;
        tc_fence_after();
        const int st = j % kStages;
        const uint32_t sb = smem_u32(smem + st * kStageBytes);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_f8_ss_if(leader, tmem + kTO + mt * kN,
                         make_sdesc(sb + mt * kAtom + kk * 4096, kAtom, 1024, SWIZZLE_128B),
                         make_sdesc(pb + kk * 32, 16, 1024, SWIZZLE_128B), idesc_pv, (j == 0 && kk == 0) ? 0u : 1u);
          }
        tc_commit_if(leader, &sm->pv_done);
        tc_commit_if(leader, &sm->kv_empty[st]);
        return true;
      };
      for (int i = 0; ok && i < nchunks; ++i) {
        const int st = i % kStages, use = i / kStages;
        if (!warp_wait(&sm->kv_full[st], use & 1, abort_flag) ||
            (i > 0 && !warp_wait(&sm->s_free, (i - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        fence_proxy_async_smem();  // the cp.async rows were written through the generic proxy
        tc_fence_after();
        const uint32_t sb = smem_u32(smem + st * kStageBytes);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          mma_f8_ss_if(leader, tmem + kTS, make_sdesc(sb + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024, SWIZZLE_128B),
                       make_sdesc(qb + (kk >> 2) * (kN * 128) + (kk & 3) * 32, 16, 1024, SWIZZLE_128B), idesc_qk,
                       kk > 0 ? 1u : 0u);
        }
        tc_commit_if(leader, &sm->s_full);
        if (i > 0 && !issue_pv(i - 1)) ok = false;
      }
      if (ok && nchunks > 0) issue_pv(nchunks - 1);
      if (leader) tc_commit(&sm->final_mma);
      __syncwarp();
      warp_wait(&sm->final_mma, 0, nullptr);
    }
  } else if (warp >= 4) {
    // ------------------------------- Q prep, softmax, epilogue (128) ----
    const int r = threadIdx.x - 128;
    const int w = warp - 4;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(w * 32) << 16);
    // exchange point of the 128 softmax threads: bounded, abort-aware mbarrier waits
    uint32_t xphase = 0;
    auto xsync = [&]() -> bool {
      warp_arrive(&sm->xchg);
      const bool ok = warp_wait(&sm->xchg, xphase & 1, abort_flag);
      ++xphase;
      return ok;
    };
    const float kv_scale = *prm.kv_scale;

    // Q: thread (head qh, eighth qj) quantises dims [64 qj, 64 qj + 64) (loaded above).
    {
      const int qh = r / 8, qj = r % 8;
      const uint4* v = qv;
      float amax = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v[c].x)), fabsf(bf16_hi(v[c].x))),
                                 fmaxf(fabsf(bf16_lo(v[c].y)), fabsf(bf16_hi(v[c].y)))));
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v[c].z)), fabsf(bf16_hi(v[c].z))),
                                 fmaxf(fabsf(bf16_lo(v[c].w)), fabsf(bf16_hi(v[c].w)))));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
      const int e = pow2_exp_448(amax);
      const float inv = exp2i(-e), qsv = exp2i(e);
      if (qj == 0) sm->qs[qh] = qsv;
      uint8_t* row = q_tile + (qj / 2) * (kN * 128) + (qh / 8) * 1024 + (qh % 8) * 128;
      uint4* erow = reinterpret_cast<uint4*>(e_tile + qh * (kD * 2) + qj * 128);
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 16 values -> one 16-byte chunk
        const uint4 a = v[2 * c], b = v[2 * c + 1];
        uint4 o;
        o.x = pack_e4m3x4(bf16_lo(a.x) * inv, bf16_hi(a.x) * inv, bf16_lo(a.y) * inv, bf16_hi(a.y) * inv);
        o.y = pack_e4m3x4(bf16_lo(a.z) * inv, bf16_hi(a.z) * inv, bf16_lo(a.w) * inv, bf16_hi(a.w) * inv);
        o.z = pack_e4m3x4(bf16_lo(b.x) * inv, bf16_hi(b.x) * inv, bf16_lo(b.y) * inv, bf16_hi(b.y) * inv);
        o.w = pack_e4m3x4(bf16_lo(b.z) * inv, bf16_hi(b.z) * inv, bf16_lo(b.w) * inv, bf16_hi(b.w) * inv);
        const int chunk = 4 * (qj % 2) + c;
        *reinterpret_cast<uint4*>(row + ((chunk ^ (qh % 8)) << 4)) = o;
        // q_hat - q of these 16 values: both have few significant bits at the
        // same scale, so the difference is exact in fp32 and in bf16
        const uint32_t code[4] = {o.x, o.y, o.z, o.w};
        const uint32_t src[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t ew[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t lo = e4m3x2_to_f16x2(code[k] & 0xFFFFu), hi = e4m3x2_to_f16x2(code[k] >> 16);
          ew[2 * k] = pack_bf16x2(f16_lo(lo) * qsv - bf16_lo(src[2 * k]), f16_hi(lo) * qsv - bf16_hi(src[2 * k]));
          ew[2 * k + 1] =
              pack_bf16x2(f16_lo(hi) * qsv - bf16_lo(src[2 * k + 1]), f16_hi(hi) * qsv - bf16_hi(src[2 * k + 1]));
        }
        erow[2 * c] = make_uint4(ew[0], ew[1], ew[2], ew[3]);
        erow[2 * c + 1] = make_uint4(ew[4], ew[5], ew[6], ew[7]);
      }
      fence_proxy_async_smem();
      warp_arrive(&sm->q_full);
    }
    bool ok = xsync();  // qs[] complete
    float c_h[kN], m_h[kN], l_h[kN];
#pragma unroll
    for (int h = 0; h < kN; ++h) {
      c_h[h] = prm.softmax_scale * kLog2e * sm->qs[h] * kv_scale;
      m_h[h] = kNegInf;
      l_h[h] = 0.f;
    }
    for (int i = 0; ok && i < nchunks; ++i) {
      const int kslot = (c0 + i) * kKeys + r;
      const bool valid = key_row(prm, t, kslot) >= 0;
      if (!warp_wait(&sm->s_full, i & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s[kN];
      tmem_ld16(lane_base + kTS, s);
      tmem_ld_wait();
      tc_fence_before();
      warp_arrive(&sm->s_free);
      float v[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) v[h] = valid ? __uint_as_float(s[h]) * c_h[h] : kNegInf;
      // per-head max over the 128 keys
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        float x = v[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        if (lane == 0) sm->red[i & 1][w][h] = x;
      }
      if (!xsync()) {
        ok = false;
        break;
      }
      float alpha[kN];
      bool any_rescale = false;
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        const float* rm = &sm->red[i & 1][0][0];
        const float mx = fmaxf(fmaxf(rm[h], rm[kN + h]), fmaxf(rm[2 * kN + h], rm[3 * kN + h]));
        alpha[h] = 1.f;
        if (mx > m_h[h] + kTau) {
          alpha[h] = ex2_approx(m_h[h] - mx);
          any_rescale |= (i > 0);
          m_h[h] = mx;
        }
      }
      uint8_t pb[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        const float msub = (m_h[h] == kNegInf) ? 0.f : m_h[h];
        const float p = ex2_approx(v[h] - msub);
        l_h[h] = l_h[h] * alpha[h] + p;
        pb[h] = static_cast<uint8_t>(pack_e4m3x2(p * kPScale, 0.f) & 0xFFu);
      }
      if (i > 0 && !warp_wait(&sm->pv_done, (i - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (any_rescale) {  // the same decision in every thread
#pragma unroll 1
        for (int mt = 0; mt < 4; ++mt) {
          uint32_t o[kN];
          tmem_ld16(lane_base + kTO + mt * kN, o);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < kN; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
          tmem_st16(lane_base + kTO + mt * kN, o);
        }
        tmem_st_wait();
      }
      // P^T tile (K-major): row h, key r
#pragma unroll
      for (int h = 0; h < kN; ++h)
        p_tile[(h / 8) * 1024 + (h % 8) * 128 + ((((r >> 4) ^ (h % 8))) << 4) + (r & 15)] = pb[h];
      fence_proxy_async_smem();
      tc_fence_before();
      warp_arrive(&sm->p_full);
    }

    if (ok && nchunks > 0 && warp_wait(&sm->pv_done, (nchunks - 1) & 1, abort_flag)) {
      tc_fence_after();
      // total row sums and final O
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        float x = l_h[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) sm->red2[w][h] = x;
      }
      ok = xsync();
      float lsum[kN], dq[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        lsum[h] = (sm->red2[0][h] + sm->red2[1][h]) + (sm->red2[2][h] + sm->red2[3][h]);
        dq[h] = 0.f;
      }
      const bool whole = prm.splits == 1;
      const size_t slot = static_cast<size_t>(t) * prm.splits + split;
      const float o_scale = kv_scale / kPScale;
      float f_h[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) f_h[h] = whole ? (lsum[h] > 0.f ? o_scale / lsum[h] : 0.f) : o_scale;
      const uint16_t* e16 = reinterpret_cast<const uint16_t*>(e_tile);
      // thread r writes dim mt * 128 + r of every head (consecutive threads, consecutive dims);
      // no branch on h_q inside the loop, so its loads and stores issue back to back
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t o[kN];
        tmem_ld16(lane_base + kTO + mt * kN, o);
        tmem_ld_wait();
        const int d = mt * 128 + r;
#pragma unroll
        for (int h = 0; h < kN; ++h) {
          const float val = __uint_as_float(o[h]) * f_h[h];
          // first-order LSE correction term: (q_hat - q) * value along this dim
          dq[h] += bf16_lo(static_cast<uint32_t>(e16[h * kD + d])) * val;
          if (h < prm.h_q) {
            if (whole)
              prm.out[(static_cast<size_t>(t) * prm.h_q + h) * kD + d] = static_cast<uint16_t>(pack_bf16x2(val, 0.f));
            else
              prm.ws_o[(slot * kN + h) * kD + d] = val;
          }
        }
      }
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        float x = dq[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) sm->red[0][w][h] = x;   // the per-step slots are no longer in use here
      }
      if (xsync() && r < prm.h_q) {
        const int h = r;
        const float dsum = (sm->red[0][0][h] + sm->red[0][1][h]) + (sm->red[0][2][h] + sm->red[0][3][h]);
        float mh = kNegInf;
#pragma unroll
        for (int k = 0; k < kN; ++k)
          if (k == h) mh = m_h[k];
        if (whole) {
          prm.lse[static_cast<size_t>(t) * prm.h_q + h] =
              lsum[h] > 0.f ? (mh + lg2_approx(lsum[h])) * kLn2 - prm.softmax_scale * dsum : kNegInf;
        } else {
          prm.ws_ml[slot * kN + h] = make_float2(lsum[h] > 0.f ? mh : kNegInf, lsum[h]);
          prm.ws_d[(slot * kN + h) * 2] = dsum;
          prm.ws_d[(slot * kN + h) * 2 + 1] = 0.f;
        }
      }
    } else if (nchunks == 0) {
      if (r < prm.h_q) {  // no key at all in this shard
        const size_t slot = static_cast<size_t>(t) * prm.splits + split;
        if (prm.splits == 1) {
          for (int d = 0; d < kD; ++d) prm.out[(static_cast<size_t>(t) * prm.h_q + r) * kD + d] = 0;
          prm.lse[static_cast<size_t>(t) * prm.h_q + r] = kNegInf;
        } else {
          prm.ws_ml[slot * kN + r] = make_float2(kNegInf, 0.f);
          prm.ws_d[(slot * kN + r) * 2] = 0.f;
          prm.ws_d[(slot * kN + r) * 2 + 1] = 0.f;
          for (int d = 0; d < kD; ++d) prm.ws_o[(slot * kN + r) * kD + d] = 0.f;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host ----

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode_rows(CUtensorMap* map, const void* base, long long rows) {
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
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {kD};
  const cuuint32_t box[2] = {128, 1};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  size_t o, ml, d, total;
};

Layout layout(int s_q, int splits) {
  const size_t slots = static_cast<size_t>(s_q) * splits;
  Layout l;
  l.o = 0;
  l.ml = round_up(slots * kN * kD * sizeof(float), 256);
  l.d = l.ml + round_up(slots * kN * sizeof(float2), 256);
  l.total = l.d + round_up(slots * kN * 2 * sizeof(float), 256);
  return l;
}

// Merge of the splits of one (token, head) row: grid (s_q, h_q), 128 threads,
// thread t owning output columns 4t .. 4t + 3.  Split j of token bi holds the
// row's fp32 partial O (true units, unnormalised) and (m, l) with m in log2
// units, plus the two LSE-correction shares d_j; the result is
// out = sum_j w_j O_j / L and lse = ln2 (M + log2 L) - scale sum_j w_j d_j / L,
// w_j = 2^(m_j - M), M = max_j m_j, L = sum_j w_j l_j, every sum in split
// order.  Up to kFewSplits splits: every thread loads every split's (m, l, d)
// (broadcast reads) together with its own partial columns and computes M, L
// and the correction itself -- one round trip, no barrier.  More splits: the
// maximum is reduced across the CTA first, then 16 splits' loads are issued
// at a time.
constexpr int kFewSplits = 16;

__global__ void __launch_bounds__(128) combine_kernel(int splits, const float* __restrict__ ws_o,
                                                      const float2* __restrict__ ws_ml,
                                                      const float* __restrict__ ws_d, float softmax_scale,
                                                      uint16_t* __restrict__ out, float* __restrict__ lse, int h_q) {
  griddep_wait();  // launched as a dependent of the decode kernel
  const int bi = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
  const size_t slot0 = static_cast<size_t>(bi) * splits;
  uint16_t* orow = out + (static_cast<size_t>(bi) * h_q + h) * kMlaDV + 4 * t;
  float* lrow = lse + static_cast<size_t>(bi) * h_q + h;
  const float2* ws_d2 = reinterpret_cast<const float2*>(ws_d);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float big_m = kNegInf, big_l = 0.f, dq = 0.f;
  auto add = [&](float w, const float4& v) {
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  };
  if (splits <= kFewSplits) {
    float4 v[kFewSplits];
    float2 ml[kFewSplits], dd[kFewSplits];
#pragma unroll
    for (int q = 0; q < kFewSplits; ++q) {
      if (q < splits) {
        const size_t slot = (slot0 + q) * kN + h;
        v[q] = __ldg(reinterpret_cast<const float4*>(ws_o + slot * kMlaDV) + t);
        ml[q] = __ldg(ws_ml + slot);
        dd[q] = __ldg(ws_d2 + slot);
      }
    }
#pragma unroll
    for (int q = 0; q < kFewSplits; ++q)
      if (q < splits) big_m = fmaxf(big_m, ml[q].x);
    if (big_m != kNegInf) {
#pragma unroll
      for (int q = 0; q < kFewSplits; ++q) {
        if (q < splits) {
          const float w = (ml[q].x == kNegInf) ? 0.f : ex2_approx(ml[q].x - big_m);  // an empty split adds nothing
          add(w, v[q]);
          big_l += w * ml[q].y;
          dq += w * (dd[q].x + dd[q].y);
        }
      }
    }
  } else {
    __shared__ float red[4];
    for (int j = t; j < splits; j += 128) big_m = fmaxf(big_m, __ldg(ws_ml + (slot0 + j) * kN + h).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) big_m = fmaxf(big_m, __shfl_xor_sync(0xffffffffu, big_m, o));
    if ((t & 31) == 0) red[t >> 5] = big_m;
    __syncthreads();
    big_m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    if (big_m != kNegInf) {
      for (int j0 = 0; j0 < splits; j0 += 16) {
        float4 v[16];
        float2 ml[16], dd[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          if (j0 + q < splits) {
            const size_t slot = (slot0 + j0 + q) * kN + h;
            v[q] = __ldg(reinterpret_cast<const float4*>(ws_o + slot * kMlaDV) + t);
            ml[q] = __ldg(ws_ml + slot);
            dd[q] = __ldg(ws_d2 + slot);
          }
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          if (j0 + q < splits) {
            const float w = (ml[q].x == kNegInf) ? 0.f : ex2_approx(ml[q].x - big_m);
            add(w, v[q]);
            big_l += w * ml[q].y;
            dq += w * (dd[q].x + dd[q].y);
          }
        }
      }
    }
  }
  if (big_m == kNegInf) {  // every split of the row is empty
    *reinterpret_cast<uint2*>(orow) = make_uint2(0, 0);
    if (t == 0) *lrow = kNegInf;
    return;
  }
  const float inv = big_l > 0.f ? 1.f / big_l : 0.f;
  *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (t == 0) *lrow = big_l > 0.f ? (big_m + lg2_approx(big_l)) * kLn2 - softmax_scale * dq * inv : kNegInf;
}

}  // namespace sparse

namespace {
// SMs of the current device (148 if it cannot be read).
int current_sms() {
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    sms = 148;
  return sms;
}

}  // namespace

int sparse_choose_splits(int s_q, int topk, int num_splits) {
  const int chunks = (topk + sparse::kKeys - 1) / sparse::kKeys;
  if (num_splits > 0) return std::min(num_splits, std::max(chunks, 1));
  const int want = std::max(1, current_sms() / std::max(s_q, 1));
  return std::max(1, std::min(want, chunks));
}

size_t sparse_workspace_bytes(int s_q, int h_q, int topk, int num_splits) {
  (void)h_q;
  if (s_q < 1 || topk < 1 || num_splits < 0) return 0;
  // the split count the decode call will choose (auto: from the current
  // device's SM count); one split writes no partials and needs no workspace
  const int splits = sparse_choose_splits(s_q, topk, num_splits);
  return splits > 1 ? sparse::layout(s_q, splits).total : 0;
}

fp8mla_status_t sparse_decode_entry(const void* q, const void* kv_cache, int64_t num_tokens, const int32_t* topk_idx,
                                    int topk, const float* kv_scale, float softmax_scale, int num_splits,
                                    void* workspace, size_t workspace_bytes, void* out, float* lse,
                                    fp8mla_dot_mode_t dot_mode, int s_q, int h_q, cudaStream_t stream) {
  if (dot_mode != FP8MLA_DOT_FP8) return FP8MLA_ERR_INVALID_ARG;  // this variant runs FP8 Q/P dots only
  if (s_q < 0 || h_q < 1 || h_q > sparse::kN || topk < 1 || num_tokens < 1 || num_splits < 0 ||
      num_tokens > (1ll << 31) - 1)
    return FP8MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f)) return FP8MLA_ERR_INVALID_ARG;
  if (s_q == 0) return FP8MLA_OK;
  if (q == nullptr || kv_cache == nullptr || topk_idx == nullptr || out == nullptr || lse == nullptr)
    return FP8MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_cache) | reinterpret_cast<uintptr_t>(out)) &
      15u)
    return FP8MLA_ERR_INVALID_ARG;
  const int splits = sparse_choose_splits(s_q, topk, num_splits);
  const sparse::Layout wl = sparse::layout(s_q, splits);
  if (splits > 1 && (workspace == nullptr || workspace_bytes < wl.total ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) ? FP8MLA_ERR_INVALID_ARG
                                                                                 : FP8MLA_ERR_WORKSPACE_TOO_SMALL;
  CUtensorMap tm;
  static TensorMapCache<8> maps;
  if (!maps.get(kv_cache, num_tokens, &tm, [&](CUtensorMap* m) { return sparse::encode_rows(m, kv_cache, num_tokens); }))
    return FP8MLA_ERR_CUDA;
  sparse::Params prm;
  char* ws = static_cast<char*>(workspace);
  prm.q = static_cast<const uint16_t*>(q);
  prm.kv = static_cast<const uint8_t*>(kv_cache);
  prm.idx = topk_idx;
  prm.kv_scale = kv_scale;
  prm.out = static_cast<uint16_t*>(out);
  prm.lse = lse;
  prm.ws_o = splits > 1 ? reinterpret_cast<float*>(ws + wl.o) : nullptr;
  prm.ws_ml = splits > 1 ? reinterpret_cast<float2*>(ws + wl.ml) : nullptr;
  prm.ws_d = splits > 1 ? reinterpret_cast<float*>(ws + wl.d) : nullptr;
  prm.num_tokens = num_tokens;
  prm.softmax_scale = softmax_scale;
  prm.topk = topk;
  prm.s_q = s_q;
  prm.h_q = h_q;
  prm.splits = splits;
  prm.chunks = (topk + sparse::kKeys - 1) / sparse::kKeys;
  static std::atomic<uint64_t> configured{0};  // per device: CUDA keeps the limit per device
  if (configure_once(configured, [] {
        return cudaFuncSetAttribute(sparse::sparse_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(sparse::kSmemBytes));
      }) != cudaSuccess)
    return FP8MLA_ERR_CUDA;
  if (launch_dependent(sparse::sparse_mla_kernel, dim3(s_q * splits), dim3(sparse::kThreads), sparse::kSmemBytes,
                       stream, tm, prm) != cudaSuccess)
    return FP8MLA_ERR_CUDA;
  if (splits > 1) {
    if (launch_dependent(sparse::combine_kernel, dim3(s_q, h_q), dim3(128), 0, stream, splits,
                         static_cast<const float*>(prm.ws_o), static_cast<const float2*>(prm.ws_ml),
                         static_cast<const float*>(prm.ws_d), softmax_scale, static_cast<uint16_t*>(out), lse,
                         h_q) != cudaSuccess)
      return FP8MLA_ERR_CUDA;
  }
  return FP8MLA_OK;
}

uint32_t sparse_read_and_clear_status() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_sparse, sizeof(v));
  cudaMemcpyToSymbol(g_status_sparse, &z, sizeof(z));
  return v;
}

}  // namespace fp8mla
