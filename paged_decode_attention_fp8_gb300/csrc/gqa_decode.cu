// Paged GQA decode over separate E4M3 K / V caches, tcgen05 + TMA, sm_103a.
//
// The operation (InfiniCore "add FP8 blockwise dequantize/GEMM operators and
// FP8(E4M3) KV cache support in paged attention": Summary, the FP8 paged
// attention decode kernel with split-kv): for batch b and query head h,
//   out[b, h] = softmax_j(scale * q[b, h] . k_j) @ v_j
// with k_j = k_scale * E4M3(K[block_table[b][j / 16], kvh, j % 16]) and v_j
// likewise from V, kvh = h / (h_q / h_kv).
//
// GB300 design (swap-AB, one CTA per (sequence, KV head, split)):
//   * 128 tokens (8 pages of 16) per step; each page's K and V tile
//     [16 tokens x 128 B] arrives by one TMA each (128-byte swizzle) into a
//     ring of three raw stages.
//   * The tensor core reads the raw E4M3 tiles: S^T = K [Q_hi | Q_lo]^T
//     (M = 128 tokens, N = 32, the K-major K tile as A: 4 MMAs) and
//     O^T = V^T [P_hi | P_lo]^T (the V tile read MN-major: 4 MMAs).  Q and P
//     enter as two E4M3 terms, hi = E4M3(x) and lo = E4M3(x - hi), about 8
//     significant bits together, side by side in one N = 32 operand: the
//     softmax adds a column's two S values, the epilogue its two O values.
//     Q carries a per-column power-of-two scale; P is stored x64 with the
//     lazy reference raised only past 2.75 (64 * 2^2.75 < 448).
//   * Softmax across TMEM lanes (one thread per token; each thread keeps
//     partial sums).  A step first votes whether any score passes its
//     column's reference by more than 2.75; only then are the per-column
//     maxima taken (shuffles + a 4-warp exchange).  Tokens
//     past the end are masked by select, and their V rows zeroed in shared
//     memory before P.V reads the tile.
//   * ~113 KB of shared memory and 128 TMEM columns per CTA: two CTAs share
//     an SM, so one's fill and drain overlap the other's steady state.
//   * Split-KV over the token dimension with a combine kernel; for small
//     grids the split count follows the FA2-style "waves" rule, the smallest
//     count within 85% of the best wave efficiency (InfiniCore page,
//     Summary: the "auto" heuristic); a grid that already fills the GPU is
//     still cut into about six CTAs per SM so unequal contexts balance,
//     unless a sliding window caps every piece (then it is not split).
//   * Per-row scales [num_blocks, h_kv, 16] (InfiniCore page, Summary): each
//     page's 16 K and 16 V scales arrive by the producer lanes' cp.async
//     with its tiles, on the same barrier; a
//     token's K scale multiplies its scores in fp32, and its V scale enters
//     the weights: u = score + log2 sigma_v, P' = 2^(u - m) carries sigma_v
//     into P.V on the raw codes, and the row sums take P' / sigma_v.
//   * XQA options (FlashInfer "add xqa fp8 mha and fp8 kv cache", launcher
//     arguments): the 16 MMA columns hold (query token, head) pairs of a
//     speculative block of q_len tokens (the last q_len cache positions),
//     masked per column by the block mask (or causally) and a sliding window
//     (steps wholly before every token's window are not loaded); sink logits
//     join the denominator once, in the epilogue or the combine.  Each option
//     set is its own kernel instance, so plain decode carries none of it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "gqa_decode.h"
#include "mla_decode.h"

namespace fp8mla {

__device__ uint32_t g_status_gqa;

namespace gqa {

constexpr int kHd = 128;
constexpr int kPage = 16;
constexpr int kTok = 128;               // tokens per step (MMA M)
constexpr int kPagesPerStep = kTok / kPage;
constexpr int kN = 16;                  // head group, padded (MMA N)
constexpr int kRawTile = kTok * kHd;    // 16 KB of E4M3 per operand per step
constexpr int kOffRawK = 0, kOffRawV = kRawTile, kRawStageBytes = 2 * kRawTile;   // 32 KB

struct Params {
  const uint16_t* q;           // bf16 [bs, q_len, h_q, 128]
  const int32_t* block_table;  // [bs, max_blocks]
  const int32_t* seqlens;      // [bs]
  const float* k_scale;        // [1], or per cached row [num_blocks, h_kv, 16] when scale_rows
  const float* v_scale;
  const uint8_t* spec_mask;    // [bs, q_len, q_len] (nonzero = visible) or null: causal inside the block
  const float* sinks;          // [h_q] sink logits or null
  uint16_t* out;               // bf16 [bs, q_len, h_q, 128]
  float* lse;                  // [bs, q_len, h_q]
  float* ws_o;                 // [bs * h_kv * splits, 16, 128]  -- indexed per (b, kv head) sequence
  float2* ws_ml;
  int num_blocks, max_blocks, bs, h_q, h_kv, group, splits;
  int q_len;                   // query tokens per sequence; MMA column n = token (n / group), head (n % group)
  int window;                  // sliding window W (0 = off): token at position p sees keys j with p - j < W
  int scale_rows;              // 1: k_scale / v_scale are per-row arrays
  float softmax_scale;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag) {
  const bool ok = wait_bounded(bar, parity, abort_flag, &g_status_gqa);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// The end of one output row: key weights summed to l against reference m (log2
// units of the scaled scores), an optional sink logit `sink` (natural units,
// -inf = none) joining the denominator once.  Returns the output factor f
// (times the accumulated P.V) and the row's LSE (natural log).  No key and no
// sink: f = 0, LSE -inf; no key with a sink: f = 0, LSE = sink.
__device__ __forceinline__ void finish_row(float m, float l, float sink, float v_scale, float* f, float* lse) {
  if (sink == kNegInf) {
    *f = l > 0.f ? v_scale / l : 0.f;
    *lse = l > 0.f ? (m + lg2_approx(l)) * kLn2 : kNegInf;
    return;
  }
  const float sk2 = sink * kLog2e;
  if (!(l > 0.f)) {
    *f = 0.f;
    *lse = sink;
    return;
  }
  const float mm = fmaxf(m, sk2);
  const float wk = ex2_approx(m - mm);
  const float den = l * wk + ex2_approx(sk2 - mm);
  *f = v_scale * wk / den;
  *lse = (mm + lg2_approx(den)) * kLn2;
}

// ------------------------------------------------------------------------
// The decode kernel: E4M3 operands straight from the TMA tiles, Q and P as two
// E4M3 terms (see the file comment).
namespace x2 {
constexpr int kThreads = 192;          // warp 0 producer, warp 1 MMA, warps 2-5 softmax and epilogue
constexpr int kStages = 3;             // raw K and V steps in flight (two CTAs per SM: six)
constexpr int kQBytes = 2 * kN * 128;  // [Q_hi ; Q_lo]: 32 rows x 128 dims E4M3, 128-byte swizzle
constexpr int kPBytes = 2 * kN * 128;  // [P_hi ; P_lo]^T: 32 rows x 128 tokens E4M3, one buffer of two
constexpr float kPScale = 64.f;
constexpr float kTau = 2.75f;          // a raised reference keeps 64 p <= 64 * 2^2.75 < 448
// TMEM: S^T (two buffers of 32 columns: hi heads 0..15, lo heads 16..31), O^T (32 columns, same split)
constexpr uint32_t kTmemCols = 128, kTS = 0, kTO = 64;

struct Smem {
  float row_scale[kStages][2][kTok];  // per-row scales of a stage's K and V rows (scale_rows)
  uint64_t raw_full[kStages], raw_empty[kStages];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];  // by step parity
  uint64_t q_full, final_mma, xchg;
  uint32_t tmem_base, abort_flag;
  float qs[kN];
  uint16_t vis_block[kN];  // per query token: bit c = key c of the speculative block visible
  // per-warp partial maxima; written only in a step whose vote passed, between that step's
  // two exchanges, so every reader of an earlier step is done with it (one buffer)
  float red[4][kN];
  float red2[4][kN];
  uint32_t grow[2][4];     // per warp: a score above its column's reference + tau (by step parity:
                           // a step without a second exchange leaves no barrier before the next vote)
};

constexpr size_t kSmemBytes = kStages * kRawStageBytes + kQBytes + 2 * kPBytes + sizeof(Smem) + 1024;
static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs fit in an SM's shared memory");

// Smallest e with amax <= 448 * 2^e (the per-head power-of-two scale of Q's hi term).
__device__ __forceinline__ int pow2_exp_448(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  const int expo = static_cast<int>((bits >> 23) & 0xFFu);
  if (expo == 0) return -126;
  const uint32_t mant = bits & 0x7FFFFFu;
  return max((expo - 127) - (mant <= 0x600000u ? 8 : 7), -126);
}
}  // namespace x2

// kG: the softmax handles MMA columns [0, kG) of the N = 16 (kG >= q_len * group).
// kMode bit 0: per-row scales; bit 1: the XQA options (q_len > 1, a mask, a window or sinks).
template <int kG, int kMode>
__global__ void __launch_bounds__(x2::kThreads, 2)
    gqa_x2_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const Params prm) {
  constexpr bool kRows = (kMode & 1) != 0, kExt = (kMode & 2) != 0;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* q_tile = smem + x2::kStages * kRawStageBytes;
  uint8_t* p_tile = q_tile + x2::kQBytes;
  x2::Smem* sm = reinterpret_cast<x2::Smem*>(p_tile + 2 * x2::kPBytes);
  volatile uint32_t* abort_flag = &sm->abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int split = blockIdx.x % prm.splits;
  const int seq = blockIdx.x / prm.splits;  // (b, kv head)
  const int b = seq / prm.h_kv;
  const int kvh = seq % prm.h_kv;

  int s_k = prm.seqlens[b];
  int n_pages = s_k > 0 ? (s_k + kPage - 1) / kPage : 0;
  if (s_k < 0 || n_pages > prm.max_blocks) {
    if (threadIdx.x == 0) atomicOr(&g_status_gqa, FP8MLA_DEV_BAD_SEQLEN);
    s_k = 0;
    n_pages = 0;
  }
  // The query block's tokens are the last q_len cache positions; with a
  // sliding window no token sees a key before k_lo, so steps wholly before it
  // are left out of the split partition.
  const int start = s_k - prm.q_len;  // position of the block's first token
  const int k_lo = (kExt && prm.window > 0) ? max(0, start - prm.window + 1) : 0;
  const int n_steps_total = (n_pages + kPagesPerStep - 1) / kPagesPerStep;
  const int step_lo = min(k_lo / kTok, n_steps_total);
  const int n_steps_all = n_steps_total - step_lo;
  const int st0 = step_lo + static_cast<int>((static_cast<long long>(split) * n_steps_all) / prm.splits);
  const int st1 = step_lo + static_cast<int>((static_cast<long long>(split + 1) * n_steps_all) / prm.splits);
  const int nsteps = st1 - st0;
  const int ncols = prm.q_len * prm.group;  // MMA columns that hold (token, head) pairs

  if (threadIdx.x == 0) {
    for (int s = 0; s < x2::kStages; ++s) {
      mbar_init(&sm->raw_full[s], kRows ? 33 : 1);  // the TMA bytes' arrival (+ per-row scales: one per lane)
      mbar_init(&sm->raw_empty[s], 1);             // the P.V that read the step's V
    }
    for (int bf = 0; bf < 2; ++bf) {
      mbar_init(&sm->s_full[bf], 1);
      mbar_init(&sm->s_free[bf], 4);
      mbar_init(&sm->p_full[bf], 4);
      mbar_init(&sm->pv_done[bf], 1);
    }
    mbar_init(&sm->q_full, 4);
    mbar_init(&sm->final_mma, 1);
    mbar_init(&sm->xchg, 4);
    sm->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm->tmem_base, x2::kTmemCols);
    tmem_relinquish();
  }
  griddep_wait();  // inputs may come from the previous kernel in the stream
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = sm->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer ----
    // lanes 0..7 fetch a step's block-table entries one step ahead; lane 0 issues the loads
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    const int32_t* bt_row = prm.block_table + static_cast<size_t>(b) * prm.max_blocks;
    auto fetch = [&](int step) {
      const int p0 = (st0 + step) * kPagesPerStep;
      return (step < nsteps && lane < min(kPagesPerStep, n_pages - p0)) ? __ldg(bt_row + p0 + lane) : 0;
    };
    int next = fetch(0);
    int i = 0;
    for (; i < nsteps; ++i) {
      const int st = i % x2::kStages, use = i / x2::kStages;
      const int p0 = (st0 + i) * kPagesPerStep;
      const int np = min(kPagesPerStep, n_pages - p0);
      int mine = next;
      next = fetch(i + 1);
      if (lane < np && (mine < 0 || mine >= prm.num_blocks)) {
        atomicOr(&g_status_gqa, FP8MLA_DEV_BAD_PAGE);
        mine = 0;
      }
      int rows[kPagesPerStep];
#pragma unroll
      for (int p = 0; p < kPagesPerStep; ++p) rows[p] = (__shfl_sync(0xffffffffu, mine, p) * prm.h_kv + kvh) * kPage;
      const int scale_row = (__shfl_sync(0xffffffffu, mine, lane / 4) * prm.h_kv + kvh) * kPage;  // page lane / 4
      bool ok = true;
      if (lane == 0) {
        ok = use == 0 || wait_bounded(&sm->raw_empty[st], (use - 1) & 1, abort_flag, &g_status_gqa);
        if (ok) {
          mbar_arrive_expect_tx(&sm->raw_full[st], 2u * np * kPage * kHd);
          uint8_t* sb = smem + st * kRawStageBytes;
#pragma unroll
          for (int p = 0; p < kPagesPerStep; ++p) {
            if (p >= np) break;
            tma_load_3d(sb + kOffRawK + p * kPage * kHd, &tm_k, &sm->raw_full[st], 0, rows[p], 0);
            tma_load_3d(sb + kOffRawV + p * kPage * kHd, &tm_v, &sm->raw_full[st], 0, rows[p], 0);
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      if constexpr (kRows) {
        // the step's row scales (rows are the scales' index too), 16 bytes a lane by cp.async
        // rather than 16 small bulk copies through the TMA unit: lane l copies scales
        // [4 (l % 4), +4) of page l / 4, of K and of V, and arrives once they land
        const int p = lane / 4, c = lane % 4;
        if (p < np) {
          cp_async16(smem_u32(&sm->row_scale[st][0][p * kPage + 4 * c]), prm.k_scale + scale_row + 4 * c, 16u);
          cp_async16(smem_u32(&sm->row_scale[st][1][p * kPage + 4 * c]), prm.v_scale + scale_row + 4 * c, 16u);
        }
        cp_async_mbar_arrive(&sm->raw_full[st]);
      }
    }
    if constexpr (kRows) cp_async_wait_all();  // this lane's copies have landed before the CTA can exit
    if (lane == 0)
      for (int j = max(0, i - x2::kStages); j < i; ++j)
        wait_bounded(&sm->raw_full[j % x2::kStages], (j / x2::kStages) & 1, nullptr, &g_status_gqa);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer ----
    // Q.K^T of step i, then P.V of step i - 1 once its P is written; the raw
    // stage of a step is released by the commit after its P.V.
    constexpr uint32_t idesc_qk = make_idesc(0, 0, 0, 0, 2 * kN, 128);  // E4M3: K (K-major) x [Q_hi|Q_lo]
    constexpr uint32_t idesc_pv = make_idesc(0, 0, 1, 0, 2 * kN, 128);  // E4M3: V^T (MN-major) x [P_hi|P_lo]^T
    const bool leader = elect_one();
    const uint32_t qb = smem_u32(q_tile);
    bool ok = warp_wait(&sm->q_full, 0, abort_flag);
    auto issue_pv = [&](int j) -> bool {
      const int bf = j & 1, st = j % x2::kStages;
      if (!warp_wait(&sm->p_full[bf], (j >> 1) & 1, abort_flag)) return false;
      tc_fence_after();
      const uint32_t vb = smem_u32(smem + st * kRawStageBytes + kOffRawV);
      const uint32_t pb = smem_u32(p_tile + bf * x2::kPBytes);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // 32 tokens per MMA
        mma_f8_ss_if(leader, tmem + x2::kTO, make_sdesc(vb + kk * 4096, kRawTile, 1024, SWIZZLE_128B),
                     make_sdesc(pb + kk * 32, 16, 1024, SWIZZLE_128B), idesc_pv, (j == 0 && kk == 0) ? 0u : 1u);
      tc_commit_if(leader, &sm->pv_done[bf]);
      tc_commit_if(leader, &sm->raw_empty[st]);
      return true;
    };
    for (int i = 0; ok && i < nsteps; ++i) {
      const int st = i % x2::kStages, bf = i & 1;
      if (!warp_wait(&sm->raw_full[st], (i / x2::kStages) & 1, abort_flag) ||
          (i >= 2 && !warp_wait(&sm->s_free[bf], ((i - 2) >> 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t kb = smem_u32(smem + st * kRawStageBytes + kOffRawK);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // 32 dims per MMA
        mma_f8_ss_if(leader, tmem + x2::kTS + bf * 2 * kN, make_sdesc(kb + kk * 32, 16, 1024, SWIZZLE_128B),
                     make_sdesc(qb + kk * 32, 16, 1024, SWIZZLE_128B), idesc_qk, kk > 0 ? 1u : 0u);
      tc_commit_if(leader, &sm->s_full[bf]);
      if (i > 0 && !issue_pv(i - 1)) ok = false;
    }
    if (ok && nsteps > 0) issue_pv(nsteps - 1);
    if (leader) tc_commit(&sm->final_mma);
    __syncwarp();
    warp_wait(&sm->final_mma, 0, nullptr);
  } else {
    // ------------------------- Q prep, softmax, epilogue (warps 2-5) ----
    const int w = warp % 4;               // TMEM lane quarter of this warp
    const int r = w * 32 + lane;          // token row of a step / TMEM lane / output dim
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(w * 32) << 16);
    uint32_t xphase = 0;
    auto xsync = [&]() -> bool {  // bounded, abort-aware exchange point of the 128 threads
      warp_arrive(&sm->xchg);
      const bool ok = warp_wait(&sm->xchg, xphase & 1, abort_flag);
      ++xphase;
      return ok;
    };
    // per-row scales enter per token (K on its scores, V through its weights)
    const float k_scale = kRows ? 1.f : *prm.k_scale, v_scale = kRows ? 1.f : *prm.v_scale;
    // column n of the MMA: query token n / group, head kvh * group + n % group
    auto q_row = [&](int n) -> const uint16_t* {
      return prm.q + ((static_cast<size_t>(b) * prm.q_len + n / prm.group) * prm.h_q + kvh * prm.group +
                      n % prm.group) * kHd;
    };
    if (kExt && r < prm.q_len) {  // which keys of the speculative block token r sees: the mask row, or c <= r
      uint32_t bits = 0;
      if (prm.spec_mask != nullptr) {
        const uint8_t* row = prm.spec_mask + (static_cast<size_t>(b) * prm.q_len + r) * prm.q_len;
        for (int c = 0; c < prm.q_len; ++c)
          if (__ldg(row + c)) bits |= 1u << c;
      } else {
        bits = (2u << r) - 1u;
      }
      sm->vis_block[r] = static_cast<uint16_t>(bits);
    }
    {
      // [Q_hi ; Q_lo]: thread (column qh, eighth qj) splits dims [16 qj, 16 qj + 16) of q / qs
      const int qh = r / 8, qj = r % 8;
      uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
      if (qh < ncols) {
        const uint16_t* qrow = q_row(qh) + qj * 16;
        v0 = __ldg(reinterpret_cast<const uint4*>(qrow));
        v1 = __ldg(reinterpret_cast<const uint4*>(qrow + 8));
      }
      const uint32_t wd[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(wd[k])), fabsf(bf16_hi(wd[k]))));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
      const int e = x2::pow2_exp_448(amax);
      const float inv = exp2i(-e);
      if (qj == 0) sm->qs[qh] = exp2i(e);
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        split_e4m3x4(bf16_lo(wd[2 * k]) * inv, bf16_hi(wd[2 * k]) * inv, bf16_lo(wd[2 * k + 1]) * inv,
                         bf16_hi(wd[2 * k + 1]) * inv, hi[k], lo[k]);
      // row n, dims [16 qj, 16 qj + 16) = 16-byte chunk qj of the 128-byte row, XOR-swizzled by n % 8
      const int nh = qh, nl = kN + qh;
      *reinterpret_cast<uint4*>(q_tile + (nh / 8) * 1024 + (nh % 8) * 128 + ((qj ^ (nh % 8)) << 4)) =
          make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(q_tile + (nl / 8) * 1024 + (nl % 8) * 128 + ((qj ^ (nl % 8)) << 4)) =
          make_uint4(lo[0], lo[1], lo[2], lo[3]);
      for (int k = r; k < 2 * x2::kPBytes / 16; k += 128) reinterpret_cast<uint4*>(p_tile)[k] = make_uint4(0, 0, 0, 0);
      fence_proxy_async_smem();
      warp_arrive(&sm->q_full);
    }
    bool ok = xsync();  // qs[], the block's visibility bits and the zeroed P tiles complete
    float c_h[kG], m_h[kG], l_h[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      c_h[h] = prm.softmax_scale * kLog2e * sm->qs[h] * k_scale;
      m_h[h] = kNegInf;
      l_h[h] = 0.f;
    }
    const uint32_t grp_bits = (1u << prm.group) - 1u;
    const bool plain = !kExt || (prm.q_len == 1 && prm.window == 0);
    for (int i = 0; ok && i < nsteps; ++i) {
      const int bf = i & 1, st = i % x2::kStages;
      const int tok = (st0 + i) * kTok + r;
      const bool live = tok < s_k;
      if (!warp_wait(&sm->s_full[bf], (i >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      // this token's K and V row scales (1 past the end: those keys are masked, and a stale
      // scale must not turn a zero weight into a NaN); the stage cannot be refilled before
      // this step's P is published, so its phase is this step's
      float sk = 1.f, lsv = 0.f, isv = 1.f;
      if constexpr (kRows) {
        if (!warp_wait(&sm->raw_full[st], (i / x2::kStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        if (live) {
          const float sv = sm->row_scale[st][1][r];
          sk = sm->row_scale[st][0][r];
          lsv = lg2_approx(sv);
          isv = 1.f / sv;
        }
      }
      tc_fence_after();
      uint32_t s[2 * kN];
      tmem_ld32(lane_base + x2::kTS + bf * 2 * kN, s);
      tmem_ld_wait();
      tc_fence_before();
      warp_arrive(&sm->s_free[bf]);
      // columns that see this thread's key: per query token ti, keys before the block always,
      // keys inside it by the token's bits, and (window W) only if ti - c_blk < W
      uint32_t colvis = 0;
      if (plain) {
        colvis = live ? 0xFFFFFFFFu : 0u;
      } else if (live) {
        const int c_blk = tok - start;
        for (int ti = 0; ti < prm.q_len; ++ti) {
          const bool vis = (c_blk < 0 || ((sm->vis_block[ti] >> c_blk) & 1u)) &&
                           (prm.window == 0 || ti - c_blk < prm.window);
          if (vis) colvis |= grp_bits << (ti * prm.group);
        }
      }
      if (!live) {  // a token past the end: zero its V row, so that P.V multiplies zeros by its zero weight
        uint4* vrow = reinterpret_cast<uint4*>(smem + st * kRawStageBytes + kOffRawV + r * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) vrow[c] = make_uint4(0, 0, 0, 0);
      }
      // (per-row scales) u = the scaled score plus log2 of the token's V scale, so that P' = 2^(u - m)
      // carries the V scale into P.V on the raw codes; the row sums take P' / sigma_v
      float v[kG];
#pragma unroll
      for (int h = 0; h < kG; ++h)
        v[h] = ((colvis >> h) & 1u) ? (__uint_as_float(s[h]) + __uint_as_float(s[kN + h])) * c_h[h] * sk + lsv
                                    : kNegInf;
      // The reference m_h of a column moves only when a score passes it by more
      // than tau, so one vote decides whether the column maxima are needed at
      // all: most steps after a CTA's first skip the per-column reductions.
      bool grow = false;
#pragma unroll
      for (int h = 0; h < kG; ++h) grow |= v[h] > m_h[h] + x2::kTau;
      grow = __any_sync(0xffffffffu, grow);
      if (lane == 0) sm->grow[i & 1][w] = grow ? 1u : 0u;
      if (!xsync()) {
        ok = false;
        break;
      }
      float alpha[kG];
      bool any_rescale = false;
#pragma unroll
      for (int h = 0; h < kG; ++h) alpha[h] = 1.f;
      if ((sm->grow[i & 1][0] | sm->grow[i & 1][1] | sm->grow[i & 1][2] | sm->grow[i & 1][3]) != 0u) {
#pragma unroll
        for (int h = 0; h < kG; ++h) {
          float x = v[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
          if (lane == 0) sm->red[w][h] = x;
        }
        if (!xsync()) {
          ok = false;
          break;
        }
#pragma unroll
        for (int h = 0; h < kG; ++h) {
          const float* rm = &sm->red[0][0];
          const float mx = fmaxf(fmaxf(rm[h], rm[kN + h]), fmaxf(rm[2 * kN + h], rm[3 * kN + h]));
          if (mx > m_h[h] + x2::kTau) {
            alpha[h] = ex2_approx(m_h[h] - mx);
            any_rescale |= (i > 0);
            m_h[h] = mx;
          }
        }
      }
      uint8_t phi[kG], plo[kG];
#pragma unroll
      for (int h = 0; h < kG; h += 4) {
        float p[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          p[k] = ex2_approx(v[h + k] - (m_h[h + k] == kNegInf ? 0.f : m_h[h + k]));
          l_h[h + k] = l_h[h + k] * alpha[h + k] + (kRows ? p[k] * isv : p[k]);
        }
        uint32_t hi, lo;
        split_e4m3x4(p[0] * x2::kPScale, p[1] * x2::kPScale, p[2] * x2::kPScale, p[3] * x2::kPScale, hi, lo);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          phi[h + k] = static_cast<uint8_t>(hi >> (8 * k));
          plo[h + k] = static_cast<uint8_t>(lo >> (8 * k));
        }
      }
      // O is rescaled only after the previous step's P.V; the P buffer is
      // rewritten only after the P.V that read it two steps ago
      if (any_rescale) {
        if (!warp_wait(&sm->pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
      } else if (i >= 2 && !warp_wait(&sm->pv_done[bf], ((i - 2) >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (any_rescale) {
        uint32_t o[2 * kN];
        tmem_ld32(lane_base + x2::kTO, o);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < kG; ++h) {
          o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
          o[kN + h] = __float_as_uint(__uint_as_float(o[kN + h]) * alpha[h]);
        }
        tmem_st32(lane_base + x2::kTO, o);
        tmem_st_wait();
      }
      // [P_hi ; P_lo]^T (K-major over tokens): row n, token r -> 16-byte chunk r / 16 (XOR n % 8), byte r % 16
      {
        uint8_t* pt = p_tile + bf * x2::kPBytes;
#pragma unroll
        for (int h = 0; h < kG; ++h) {
          const int nl = kN + h;
          pt[(h / 8) * 1024 + (h % 8) * 128 + (((r >> 4) ^ (h % 8)) << 4) + (r & 15)] = phi[h];
          pt[(nl / 8) * 1024 + (nl % 8) * 128 + (((r >> 4) ^ (nl % 8)) << 4) + (r & 15)] = plo[h];
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      warp_arrive(&sm->p_full[bf]);
    }

    const bool whole = prm.splits == 1;
    const size_t slot = static_cast<size_t>(seq) * prm.splits + split;
    const float o_scale = v_scale / x2::kPScale;
    if (ok && nsteps > 0 && warp_wait(&sm->pv_done[(nsteps - 1) & 1], ((nsteps - 1) >> 1) & 1, abort_flag)) {
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        float x = l_h[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) sm->red2[w][h] = x;
      }
      ok = xsync();
      uint32_t o[2 * kN];
      tmem_ld32(lane_base + x2::kTO, o);
      tmem_ld_wait();
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        if (h >= ncols) break;
        const float lsum = (sm->red2[0][h] + sm->red2[1][h]) + (sm->red2[2][h] + sm->red2[3][h]);
        const float oh = __uint_as_float(o[h]) + __uint_as_float(o[kN + h]);
        const int hq = kvh * prm.group + h % prm.group;
        const size_t orow = (static_cast<size_t>(b) * prm.q_len + h / prm.group) * prm.h_q + hq;
        if (whole) {
          float f, lse_v;
          finish_row(m_h[h], lsum, (kExt && prm.sinks) ? prm.sinks[hq] : kNegInf, o_scale, &f, &lse_v);
          prm.out[orow * kHd + r] = static_cast<uint16_t>(pack_bf16x2(oh * f, 0.f));
          if (r == 0) prm.lse[orow] = lse_v;
        } else {
          prm.ws_o[(slot * kN + h) * kHd + r] = oh * o_scale;
          if (r == 0) prm.ws_ml[slot * kN + h] = make_float2(lsum > 0.f ? m_h[h] : kNegInf, lsum);
        }
      }
    } else if (ok && nsteps == 0) {
      for (int h = 0; h < ncols; ++h) {
        const int hq = kvh * prm.group + h % prm.group;
        const size_t orow = (static_cast<size_t>(b) * prm.q_len + h / prm.group) * prm.h_q + hq;
        if (whole) {  // no key: out 0, lse the sink's logit (-inf without one)
          prm.out[orow * kHd + r] = 0;
          if (r == 0) prm.lse[orow] = (kExt && prm.sinks) ? prm.sinks[hq] : kNegInf;
        } else {
          prm.ws_o[(slot * kN + h) * kHd + r] = 0.f;
          if (r == 0) prm.ws_ml[slot * kN + h] = make_float2(kNegInf, 0.f);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, x2::kTmemCols);
  }
}

// Merge of split partials: one warp per (sequence = (b, kv head), column = (token, head)), lane l owns
// 4 dims; a sink logit joins the merged denominator once.
__global__ void gqa_combine_kernel(const float* __restrict__ ws_o, const float2* __restrict__ ws_ml, int splits,
                                   int group, int q_len, int h_q, int h_kv, const float* __restrict__ sinks,
                                   uint16_t* __restrict__ out, float* __restrict__ lse) {
  griddep_wait();  // launched as a dependent of the decode kernel
  const int seq = blockIdx.x;
  const int h = blockIdx.y * 4 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (h >= q_len * group) return;
  const int b = seq / h_kv, kvh = seq % h_kv;
  const int hq = kvh * group + h % group;
  const size_t row = (static_cast<size_t>(b) * q_len + h / group) * h_q + hq;
  const float sink = sinks ? sinks[hq] : kNegInf;
  float big_m = kNegInf;
  for (int s = 0; s < splits; ++s) big_m = fmaxf(big_m, ws_ml[(static_cast<size_t>(seq) * splits + s) * kN + h].x);
  uint16_t* orow = out + row * kHd + lane * 4;
  if (big_m == kNegInf) {  // no key: out 0, lse the sink's logit (-inf without one)
    *reinterpret_cast<uint2*>(orow) = make_uint2(0, 0);
    if (lane == 0) lse[row] = sink;
    return;
  }
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, big_l = 0.f;
  for (int s = 0; s < splits; ++s) {
    const size_t slot = (static_cast<size_t>(seq) * splits + s) * kN + h;
    const float2 ml = ws_ml[slot];
    if (ml.x == kNegInf) continue;
    const float wgt = ex2_approx(ml.x - big_m);
    big_l += ml.y * wgt;
    const float4 v = *reinterpret_cast<const float4*>(ws_o + slot * kHd + lane * 4);
    acc[0] += wgt * v.x;
    acc[1] += wgt * v.y;
    acc[2] += wgt * v.z;
    acc[3] += wgt * v.w;
  }
  float inv, lse_v;
  finish_row(big_m, big_l, sink, 1.f, &inv, &lse_v);
  *reinterpret_cast<uint2*>(orow) =
      make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
  if (lane == 0) lse[row] = lse_v;
}

// ---------------------------------------------------------------- host ----

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 3-D view {128 B, rows, 1} of a cache as [num_blocks * h_kv * 16] rows of 128 bytes, box = one page.
bool encode_pages(CUtensorMap* map, const void* base, long long rows) {
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
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHd), static_cast<cuuint64_t>(rows), 1};
  const cuuint64_t strides[2] = {kHd, static_cast<cuuint64_t>(rows) * kHd};
  const cuuint32_t box[3] = {128, kPage, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace gqa

namespace {
// The fewest splits whose grid of ctas * s CTAs fills its waves of num_sms to
// within 85 % of the best fill over 1 .. cap splits.
int waves_rule(long long ctas, int cap, int num_sms) {
  double eff[17] = {0}, best = 0;
  for (int s = 1; s <= cap; ++s) {
    const long long n = ctas * s;
    const long long waves = (n + num_sms - 1) / num_sms;
    eff[s] = static_cast<double>(n) / static_cast<double>(waves * num_sms);
    best = std::max(best, eff[s]);
  }
  for (int s = 1; s <= cap; ++s)
    if (eff[s] >= 0.85 * best) return s;
  return 1;
}
}  // namespace

int gqa_choose_splits(int bs, int h_kv, int max_seqlen, int num_sms, int num_splits, bool capped) {
  const int max_steps = std::max(1, (max_seqlen + gqa::kTok - 1) / gqa::kTok);
  if (num_splits > 0) return std::max(1, std::min(num_splits, max_steps));
  const long long ctas = static_cast<long long>(std::max(bs, 1)) * std::max(h_kv, 1);
  if (num_sms < 1) return 1;
  const int cap = std::min(16, max_steps);
  if (ctas * 5 >= static_cast<long long>(num_sms) * 4) {
    // The grid already fills the GPU.  A window caps every sequence's keys,
    // so the (sequence, KV head) pieces are nearly equal and splitting them
    // only adds fill, drain and a merge (bs = 32, h_kv = 8, a 4096-key
    // window: 58 us with 1 split, 69 with 2, 84 with 4).  Without one,
    // contexts of unequal length leave the last wave ragged: cut every
    // sequence into a few pieces (about six CTAs per SM, each of at least 8
    // steps) so the hardware scheduler can balance.
    if (capped) return 1;
    const long long want = (6LL * num_sms + ctas - 1) / ctas;
    return static_cast<int>(std::max(1LL, std::min({want, 16LL, static_cast<long long>(max_steps / 8)})));
  }
  return waves_rule(ctas, cap, num_sms);
}

size_t gqa_workspace_bytes(int bs, int h_q, int head_dim, int max_splits) {
  (void)h_q;
  if (bs < 1 || max_splits < 2 || head_dim != gqa::kHd) return 0;
  // slots: every (b, kv head) pair needs max_splits slots of 16 heads; h_kv <= h_q bounds the pairs
  const size_t slots = static_cast<size_t>(bs) * std::max(h_q, 1) * max_splits;
  return gqa::round_up(slots * gqa::kN * gqa::kHd * sizeof(float), 256) +
         gqa::round_up(slots * gqa::kN * sizeof(float2), 256);
}

fp8mla_status_t gqa_decode_entry(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                 const float* k_scale, const float* v_scale, int scale_rows,
                                 const int32_t* block_table, int max_blocks, const int32_t* seqlens,
                                 float softmax_scale, int q_len, const uint8_t* spec_mask, int window,
                                 const float* sinks, int num_splits, void* workspace, size_t workspace_bytes,
                                 void* out, float* lse, int bs, int h_q, int h_kv, int head_dim, int page_size,
                                 cudaStream_t stream) {
  if (head_dim != gqa::kHd || page_size != gqa::kPage || bs < 0 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0 ||
      q_len < 1 || static_cast<long long>(q_len) * (h_q / h_kv) > gqa::kN || window < 0 || num_blocks < 1 ||
      max_blocks < 1 || num_splits < 0 || !(softmax_scale > 0.f))
    return FP8MLA_ERR_INVALID_ARG;
  if (bs == 0) return FP8MLA_OK;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr || seqlens == nullptr ||
      out == nullptr || lse == nullptr)
    return FP8MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache)) & 15u)
    return FP8MLA_ERR_INVALID_ARG;
  // per-row scales arrive by 64-byte bulk copies
  if (scale_rows && ((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) & 15u))
    return FP8MLA_ERR_INVALID_ARG;
  int splits = std::min(num_splits, 1 << 16);
  if (splits == 0) {  // auto: the waves rule for this GPU, with the block table's capacity as the longest
                      // context (or, with a window, the keys a window spans plus one step of alignment)
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
      return FP8MLA_ERR_CUDA;
    long long longest = static_cast<long long>(max_blocks) * gqa::kPage;
    if (window > 0) longest = std::min(longest, static_cast<long long>(window) + q_len - 1 + gqa::kTok);
    splits = gqa_choose_splits(bs, h_kv, static_cast<int>(longest), sms, 0, window > 0);
  }
  if (splits > 1) {
    const size_t need = gqa_workspace_bytes(bs, h_q, head_dim, splits);
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FP8MLA_ERR_INVALID_ARG;
    if (workspace_bytes < need) return FP8MLA_ERR_WORKSPACE_TOO_SMALL;
  }
  const long long rows = static_cast<long long>(num_blocks) * h_kv * gqa::kPage;
  CUtensorMap tk, tv;
  static TensorMapCache<16> maps;
  if (!maps.get(k_cache, rows, &tk, [&](CUtensorMap* m) { return gqa::encode_pages(m, k_cache, rows); }) ||
      !maps.get(v_cache, rows, &tv, [&](CUtensorMap* m) { return gqa::encode_pages(m, v_cache, rows); }))
    return FP8MLA_ERR_CUDA;
  gqa::Params prm;
  prm.q = static_cast<const uint16_t*>(q);
  prm.block_table = block_table;
  prm.seqlens = seqlens;
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  prm.scale_rows = scale_rows ? 1 : 0;
  prm.spec_mask = spec_mask;
  prm.sinks = sinks;
  prm.q_len = q_len;
  prm.window = window;
  prm.out = static_cast<uint16_t*>(out);
  prm.lse = lse;
  const size_t slots = static_cast<size_t>(bs) * h_kv * splits;
  prm.ws_o = splits > 1 ? static_cast<float*>(workspace) : nullptr;
  prm.ws_ml = splits > 1 ? reinterpret_cast<float2*>(static_cast<char*>(workspace) +
                                                     gqa::round_up(slots * gqa::kN * gqa::kHd * sizeof(float), 256))
                         : nullptr;
  prm.num_blocks = num_blocks;
  prm.max_blocks = max_blocks;
  prm.bs = bs;
  prm.h_q = h_q;
  prm.h_kv = h_kv;
  prm.group = h_q / h_kv;
  prm.splits = splits;
  prm.softmax_scale = softmax_scale;
  // one kernel instance per (option set, column count): kMode bit 0 per-row scales, bit 1 the XQA options
  using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const gqa::Params);
  static const KernelFn table[4][3] = {
      {gqa::gqa_x2_kernel<4, 0>, gqa::gqa_x2_kernel<8, 0>, gqa::gqa_x2_kernel<16, 0>},
      {gqa::gqa_x2_kernel<4, 1>, gqa::gqa_x2_kernel<8, 1>, gqa::gqa_x2_kernel<16, 1>},
      {gqa::gqa_x2_kernel<4, 2>, gqa::gqa_x2_kernel<8, 2>, gqa::gqa_x2_kernel<16, 2>},
      {gqa::gqa_x2_kernel<4, 3>, gqa::gqa_x2_kernel<8, 3>, gqa::gqa_x2_kernel<16, 3>}};
  static std::atomic<uint64_t> configured{0};  // per device: CUDA keeps the limit per device
  if (configure_once(configured, [] {
        cudaError_t e = cudaSuccess;
        for (const auto& row : table)
          for (KernelFn f : row)
            if (e == cudaSuccess)
              e = cudaFuncSetAttribute(reinterpret_cast<const void*>(f), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(gqa::x2::kSmemBytes));
        return e;
      }) != cudaSuccess)
    return FP8MLA_ERR_CUDA;
  const long long grid = static_cast<long long>(bs) * h_kv * splits;
  if (grid > 0x7FFFFFFFll) return FP8MLA_ERR_INVALID_ARG;
  const int ncols = q_len * prm.group;
  const bool ext = q_len > 1 || window > 0 || spec_mask != nullptr || sinks != nullptr;
  const int mode = (scale_rows ? 1 : 0) | (ext ? 2 : 0);
  const int gi = ncols <= 4 ? 0 : (ncols <= 8 ? 1 : 2);
  const cudaError_t le = launch_dependent(table[mode][gi], dim3(static_cast<unsigned>(grid)),
                                          dim3(gqa::x2::kThreads), gqa::x2::kSmemBytes, stream, tk, tv, prm);
  if (le != cudaSuccess) return FP8MLA_ERR_CUDA;
  if (splits > 1) {
    dim3 cg(static_cast<unsigned>(bs * h_kv), (ncols + 3) / 4);
    if (launch_dependent(gqa::gqa_combine_kernel, cg, dim3(128), 0, stream, prm.ws_o, prm.ws_ml, splits, prm.group,
                         q_len, h_q, h_kv, sinks, prm.out, lse) != cudaSuccess)
      return FP8MLA_ERR_CUDA;
  }
  return FP8MLA_OK;
}

uint32_t gqa_read_and_clear_status() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_gqa, sizeof(v));
  cudaMemcpyToSymbol(g_status_gqa, &z, sizeof(z));
  return v;
}

}  // namespace fp8mla
