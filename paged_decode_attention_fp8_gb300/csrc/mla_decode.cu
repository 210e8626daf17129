// Dense MLA decode over an E4M3 paged KV cache, tcgen05 + TMA, sm_103a.
//
// The operation (FlashMLA "update fp8 support", Improvements; test shape
// d = 576, dv = 512, h_kv = 1, s_q <= 2, causal) per sequence b:
//   S = Q K^T (Q: R = s_q * h_q rows x 576; K: the sequence's cached rows),
//   P = softmax(softmax_scale * S) under the causal mask, O = P V with V the
//   first 512 dims of the same rows; lse = log sum exp.
//
// GB300 design: one work unit = 2 CTAs (FP8 dots, mla_fp8_kernel) or 4 CTAs
// (16-bit dots, mla_decode_16bit_kernel), each owning one slice of dv.
//   * TMA loads a whole 64-token page through the block table: four
//     128-byte-swizzled boxes of the 512 latent bytes (usable as K-major B
//     for Q.K^T and as MN-major B for P.V without any transpose) and one
//     plain box of the 64 RoPE bytes.
//   * FP8 dots: Q is quantised by mla_qprep_kernel one grid ahead (per-row
//     power-of-two scale qs; latent -> E4M3, RoPE -> f16 divided by qs
//     exactly; aiter sparse_mla_fwd page, Technical details: Q quantisation)
//     and carried through the page ring.  TMEM holds O (256 columns), two S
//     buffers (64 each; pages alternate) and the latent Q (128, the A operand
//     of the latent Q.K^T); shared memory holds the ring, the page's RoPE part
//     converted to f16 (exact for E4M3), the Q RoPE tile and the P tile.
//     Q.K^T = 16 E4M3 MMAs (K = 32) + 4 f16 MMAs (K = 16) into one f32
//     accumulator -- the RoPE chunk stays 16-bit (FlashMLA page,
//     Improvements) -- and P.V = 2 E4M3 MMAs with N = 256.
//   * 16-bit dots: converter warps turn each page into bf16 (exact); Q, S, P
//     and O live in TMEM and both products run as bf16 MMAs.
//   * Online softmax in the log2 domain (InfiniCore page, Summary) with the
//     per-tensor kv_scale and qs folded into one per-row constant; with FP8
//     dots P is stored as E4M3(64 p) so long tails do not flush to zero, and
//     the running max is only raised when a page's max exceeds it by more
//     than 2.75 (log2 units): 64 p <= 64 * 2^2.75 < 448 and O rescales are
//     rare (aiter page, Technical details and Accuracy).
//   * Rows of the sequence's last page past its length are zeroed once per
//     sequence before P.V reads them (FlashMLA page, TODO: fill_oob_KV per
//     tile was the stated limiter); scores there are masked by a select.
//   * A unit may cover a piece of a sequence; pieces publish (m, l, O) to a
//     workspace and a combine kernel merges them (InfiniCore split-kv commit).
//   * FP8 dots perturb the LSE by softmax_scale * (q_hat - q) . k_mean, where
//     k_mean = sum_j p_j k_j; its latent part is exactly the output row, so
//     the combine kernel subtracts softmax_scale * (q_hat - q) . out, from the
//     quantisation error the prep kernel stored and the finished output row.
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-3 page conversion (the RoPE part to f16, or the whole page
// to bf16) and tail zeroing, warps 4-11 softmax, Q copy and epilogue: query
// row r (= TMEM lane r) is shared by two threads, each owning half of the
// page's score columns and half of the O slice.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "common.cuh"
#include "mla_decode.h"

namespace fp8mla {

__device__ uint32_t g_status_mla;

namespace mla {

constexpr int kPage = 64;
constexpr int kD = 576;
constexpr int kDLat = 512;
constexpr int kDV = 512;
constexpr int kRows = 128;
constexpr int kSoftmaxThreads = 256;                // two threads per query row
constexpr int kLatBox = kPage * 128;                 // one 128-byte column slice of a page (8 KB)
constexpr uint32_t kPageTxBytes = kPage * kD;        // bytes one page's TMA loads deliver

// 16-bit dots (exact): 4 CTAs per unit, each owning a 128-column slice of dv.
struct Cfg16 {
  static constexpr int kParts = 4, kDvPart = 128, kStages = 2;
  static constexpr int kThreads = 384;
  static constexpr float kPScale = 1.0f, kPLog2 = 0.0f, kTau = 8.0f;
  static constexpr int kOffRope8 = 4 * kLatBox;
  static constexpr int kOffCvt = kOffRope8 + kPage * 64;  // 9 bf16 boxes: 8 latent + RoPE
  static constexpr int kStageBytes = kOffCvt + 9 * kLatBox;
  static constexpr uint32_t kTO = 0, kTS = 128, kTP = 192, kTQ = 224, kTQR = 224 + 256;
};
static_assert(Cfg16::kOffCvt % 1024 == 0 && Cfg16::kStageBytes % 1024 == 0, "1 KB aligned tiles");

struct Barriers16 {
  uint64_t kv_full[Cfg16::kStages];
  uint64_t kv_empty[Cfg16::kStages];
  uint64_t cvt_ready[Cfg16::kStages];
  uint64_t s_full, s_free, p_full, pv_done, q_full, final_mma;
  uint64_t xchg;            // softmax-group exchange barrier (all 256 softmax threads arrive)
  uint32_t tmem_base;
  uint32_t abort_flag;
  uint32_t cvt_ok;
  float xmax[2][2][kRows];  // per-page tile max of each row half, double-buffered by page parity
  float xsum[2][kRows];     // row-sum halves
};

constexpr size_t smem_bytes16() { return Cfg16::kStages * Cfg16::kStageBytes + sizeof(Barriers16) + 1024; }

// One (sequence, page range) piece of a unit's work.
struct Segment {
  int b, lo, hi, split, s_k, n;
};

// Walks the segments of one unit: sequences b_begin .. b_end of the tile
// schedule, clipped to the unit's page range, skipping empty pieces.
struct SegmentWalker {
  int b, b0, p0, b1, p1, k0;
  const MlaParams* prm;
  __device__ SegmentWalker(const MlaParams& p, int unit) : prm(&p) {
    const int32_t* row = p.tile_sched + unit * 8;
    b0 = row[0];
    p0 = row[1];
    b1 = row[2];
    p1 = row[3];
    k0 = row[4];
    b = b0;
  }
  __device__ bool next(Segment& s) {
    while (b <= b1 && b < prm->b) {
      const int bb = b++;
      const int s_k = prm->seqlens[bb];
      const int n = seq_pages(s_k, kPage, prm->max_pages, &g_status_mla);
      const int lo = (bb == b0) ? p0 : 0;
      int hi = (bb == b1) ? p1 : n;
      hi = min(hi, n);
      if (hi <= lo) continue;
      s = Segment{bb, lo, hi, (bb == b0) ? k0 : 0, s_k, n};
      return true;
    }
    return false;
  }
};

// site: a source line recorded if the wait runs out
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          uint32_t site = 0) {
  const bool ok = wait_bounded<kCluster>(bar, parity, abort_flag, &g_status_mla, site);
  return __all_sync(0xffffffffu, ok);
}

// warp_wait polling without suspension, for the waits on the per-page critical path
template <bool kCluster = false>
__device__ __forceinline__ bool warp_spin(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          uint32_t site = 0) {
  const bool ok = wait_spin<kCluster>(bar, parity, abort_flag, &g_status_mla, site);
  return __all_sync(0xffffffffu, ok);
}

// Smallest e with amax <= 448 * 2^e (exact, from the float's exponent and mantissa).
__device__ __forceinline__ int pow2_scale_exponent(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  const int expo = static_cast<int>((bits >> 23) & 0xFFu);
  if (expo == 0) return -126;  // zero or subnormal: any scale in range works
  const uint32_t mant = bits & 0x7FFFFFu;
  const int e = (expo - 127) - (mant <= 0x600000u ? 8 : 7);  // 448 = 1.75 * 2^8
  return max(e, -126);
}

__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

__device__ __forceinline__ float absmax_bf16x8(uint4 v) {
  return fmaxf(fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))), fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)))),
               fmaxf(fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))), fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w)))));
}

// Dense MLA decode with 16-bit dots: Q and every page converted to bf16
// (exact), bf16 MMAs; the reference for the FP8-dot kernel's rounding.
__global__ void __launch_bounds__(Cfg16::kThreads, 1)
    mla_decode_16bit_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope,
                            const MlaParams prm) {
  using C = Cfg16;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  Barriers16* bars = reinterpret_cast<Barriers16*>(smem + C::kStages * C::kStageBytes);
  volatile uint32_t* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int unit = blockIdx.x / C::kParts;
  const int part = blockIdx.x % C::kParts;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
      mbar_init(&bars->cvt_ready[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, kSoftmaxThreads / 32);   // one arrival per softmax warp
    mbar_init(&bars->p_full, kSoftmaxThreads / 32);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->q_full, kSoftmaxThreads / 32);
    mbar_init(&bars->final_mma, 1);
    mbar_init(&bars->xchg, kSoftmaxThreads / 32);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  // Everything above overlaps the previous kernel (launched as its dependent);
  // from here on this grid reads the schedule and writes outputs.
  griddep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = bars->tmem_base;


  if (warp == 0) {
    // ------------------------------------------------ TMA producer ----
    // The warp loads 32 block-table entries at a time (one per lane) and lane 0
    // issues the page loads, so no page waits on its own table lookup.
    if (lane == 0) {
      tma_prefetch_desc(&tm_lat);
      tma_prefetch_desc(&tm_rope);
    }
    SegmentWalker walk(prm, unit);
    Segment sg;
    int i = 0;
    bool ok = true;
    while (ok && walk.next(sg)) {
      const int32_t* bt = prm.block_table + static_cast<size_t>(sg.b) * prm.max_pages;
      for (int chunk = sg.lo; ok && chunk < sg.hi; chunk += 32) {
        int mine = 0;
        if (chunk + lane < sg.hi) {
          mine = __ldg(bt + chunk + lane);
          if (mine < 0 || mine >= prm.num_pages) {
            atomicOr(&g_status_mla, FP8MLA_DEV_BAD_PAGE);
            mine = 0;
          }
        }
        const int cnt = min(32, sg.hi - chunk);
        for (int j = 0; j < cnt; ++j, ++i) {
          const int phys = __shfl_sync(0xffffffffu, mine, j);
          const int st = i % C::kStages;
          const int use = i / C::kStages;
          bool waited = true;
          if (lane == 0) {
            waited = use == 0 || wait_bounded(&bars->kv_empty[st], (use - 1) & 1, abort_flag, &g_status_mla, __LINE__);
            if (waited) {
              uint8_t* sb = smem + st * C::kStageBytes;
              mbar_arrive_expect_tx(&bars->kv_full[st], kPageTxBytes);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                tma_load_3d(sb + k * kLatBox, &tm_lat, &bars->kv_full[st], k * 128, 0, phys);
              tma_load_3d(sb + C::kOffRope8, &tm_rope, &bars->kv_full[st], kDLat, 0, phys);
            }
          }
          if (!__shfl_sync(0xffffffffu, waited ? 1 : 0, 0)) {
            ok = false;
            break;
          }
        }
      }
    }
    // Never leave with copies in flight: wait for the last loads issued.
    if (lane == 0)
      for (int j = max(0, i - C::kStages); j < i; ++j)
        wait_bounded(&bars->kv_full[j % C::kStages], (j / C::kStages) & 1, nullptr, &g_status_mla, __LINE__);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer ----
    if (lane == 0) {
      const uint32_t t_s = tmem + C::kTS, t_o = tmem + C::kTO;
      SegmentWalker walk(prm, unit);
      Segment sg;
      int i = 0, seg_i = 0;
      bool ok = true;

      auto issue_qk = [&](uint32_t sb) {
        {
          constexpr uint32_t idesc16 = make_idesc(1, 1, 0, 0, 64, 128);
#pragma unroll
          for (int kk = 0; kk < 36; ++kk) {
            const uint64_t bd =
                make_sdesc(sb + C::kOffCvt + (kk >> 2) * kLatBox + (kk & 3) * 32, 16, 1024, SWIZZLE_128B);
            mma_f16_ts(t_s, tmem + C::kTQ + kk * 8, bd, idesc16, kk > 0 ? 1u : 0u);
          }
        }
      };

      auto issue_pv = [&](int j, bool first_in_seg) -> bool {
        if (!wait_bounded(&bars->p_full, j & 1, abort_flag, &g_status_mla, __LINE__)) return false;
        tc_fence_after();
        const int st = j % C::kStages;
        const uint32_t sb = smem_u32(smem + st * C::kStageBytes);
        {
          constexpr uint32_t idesc = make_idesc(1, 1, 0, 1, 128, 128);   // bf16, B MN-major, N = 128
          const uint32_t v_base = sb + C::kOffCvt + part * 2 * kLatBox;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = make_sdesc(v_base + kk * 2048, kLatBox, 1024, SWIZZLE_128B);
            mma_f16_ts(t_o, tmem + C::kTP + kk * 8, bd, idesc, (first_in_seg && kk == 0) ? 0u : 1u);
          }
        }
        tc_commit(&bars->pv_done);
        tc_commit(&bars->kv_empty[st]);
        return true;
      };

      while (ok && walk.next(sg)) {
        if (!wait_bounded(&bars->q_full, seg_i & 1, abort_flag, &g_status_mla, __LINE__)) break;
        const int first_i = i;
        for (int pg = sg.lo; pg < sg.hi; ++pg, ++i) {
          const int st = i % C::kStages;
          const int use = i / C::kStages;
          if (!wait_bounded(&bars->kv_full[st], use & 1, abort_flag, &g_status_mla, __LINE__) ||
              !wait_bounded(&bars->cvt_ready[st], use & 1, abort_flag, &g_status_mla, __LINE__) ||
              (i > 0 && !wait_bounded(&bars->s_free, (i - 1) & 1, abort_flag, &g_status_mla, __LINE__))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_qk(smem_u32(smem + st * C::kStageBytes));
          tc_commit(&bars->s_full);
          if (i > first_i && !issue_pv(i - 1, i - 1 == first_i)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        if (!issue_pv(i - 1, i - 1 == first_i)) break;
        ++seg_i;
      }
      tc_commit(&bars->final_mma);
      wait_bounded(&bars->final_mma, 0, nullptr, &g_status_mla, __LINE__);
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    // ------------------------------- page conversion, tail zeroing ----
    const int t = threadIdx.x - 64;  // token row of the page
    SegmentWalker walk(prm, unit);
    Segment sg;
    int i = 0;
    bool ok = true;
    while (ok && walk.next(sg)) {
      for (int pg = sg.lo; pg < sg.hi; ++pg, ++i) {
        const int st = i % C::kStages;
        const int use = i / C::kStages;
        if (t == 0) bars->cvt_ok = wait_bounded(&bars->kv_full[st], use & 1, abort_flag, &g_status_mla, __LINE__) ? 1u : 0u;
        named_bar_sync(1, 64);
        if (!bars->cvt_ok) {
          ok = false;
          break;
        }
        uint8_t* sb = smem + st * C::kStageBytes;
        const bool dead = (pg == sg.n - 1) && (t >= sg.s_k - pg * kPage);  // slot past the sequence end
        const uint4 z = make_uint4(0, 0, 0, 0);
        const int sw = t & 7;
        // RoPE bytes -> bf16 (box C::kOffCvt + (8 boxes))
        {
          const uint4* src = reinterpret_cast<const uint4*>(sb + C::kOffRope8 + t * 64);
          uint8_t* dst = sb + C::kOffCvt + 8 * kLatBox + t * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4 lo = z, hi = z;
            if (!dead) {
              const uint4 v = src[c];
              e4m3x4_to_bf16x4(v.x, lo.x, lo.y);
              e4m3x4_to_bf16x4(v.y, lo.z, lo.w);
              e4m3x4_to_bf16x4(v.z, hi.x, hi.y);
              e4m3x4_to_bf16x4(v.w, hi.z, hi.w);
            }
            *reinterpret_cast<uint4*>(dst + (((2 * c) ^ sw) << 4)) = lo;
            *reinterpret_cast<uint4*>(dst + (((2 * c + 1) ^ sw) << 4)) = hi;
          }
        }
        {
          // latent: raw box j chunk c (16 E4M3) -> bf16 box 2j + c/4, chunks 2(c%4), 2(c%4)+1
#pragma unroll 1
          for (int j = 0; j < 4; ++j) {
            const uint8_t* src = sb + j * kLatBox + t * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint4 lo = z, hi = z;
              if (!dead) {
                const uint4 v = *reinterpret_cast<const uint4*>(src + ((c ^ sw) << 4));
                e4m3x4_to_bf16x4(v.x, lo.x, lo.y);
                e4m3x4_to_bf16x4(v.y, lo.z, lo.w);
                e4m3x4_to_bf16x4(v.z, hi.x, hi.y);
                e4m3x4_to_bf16x4(v.w, hi.z, hi.w);
              }
              uint8_t* dst = sb + C::kOffCvt + (2 * j + c / 4) * kLatBox + t * 128;
              *reinterpret_cast<uint4*>(dst + (((2 * (c % 4)) ^ sw) << 4)) = lo;
              *reinterpret_cast<uint4*>(dst + (((2 * (c % 4) + 1) ^ sw) << 4)) = hi;
            }
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 64);
        if (t == 0) mbar_arrive(&bars->cvt_ready[st]);
      }
    }
  } else {
    // ------------------ softmax / Q prep / epilogue (8 warps, 2 per row) ----
    const int hf = (warp - 4) / 4;                          // which half of the row
    const int r = (warp % 4) * 32 + lane;                   // query row = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    const float kv_scale = *prm.kv_scale;
    const int R = prm.s_q * prm.h_q;
    constexpr int kOHalf = C::kDvPart / 2;                  // O columns of this thread
    // Exchange point of the 256 softmax threads: an mbarrier with bounded,
    // abort-aware waits, so no thread can block forever on a peer that stopped.
    uint32_t xphase = 0;
    auto xsync = [&]() -> bool {
      warp_arrive(&bars->xchg);
      const bool ok = warp_wait(&bars->xchg, xphase & 1, abort_flag, __LINE__);
      ++xphase;
      return ok;
    };
    SegmentWalker walk(prm, unit);
    Segment sg;
    int i = 0;
    while (walk.next(sg)) {
      const uint16_t* qrow = prm.q + (static_cast<size_t>(sg.b) * R + r) * kD;
      float c_row;
      {
        // ---- Q preparation: bf16 as is; 64-value chunks 0-4 (hf 0) or 5-8 (hf 1) ----
        c_row = prm.softmax_scale * kLog2e * kv_scale;
#pragma unroll 1
        for (int ch = hf ? 5 : 0; ch < (hf ? 9 : 5); ++ch) {
          uint32_t pk[32];
          const uint4* q4 = reinterpret_cast<const uint4*>(qrow + ch * 64);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < R) v = __ldg(q4 + c);
            pk[4 * c + 0] = v.x;
            pk[4 * c + 1] = v.y;
            pk[4 * c + 2] = v.z;
            pk[4 * c + 3] = v.w;
          }
          tmem_st32(lane_base + C::kTQ + ch * 32, pk);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(&bars->q_full);
      {  // warm L2 with the next segment's Q rows while this one runs
        SegmentWalker peek = walk;
        Segment nx;
        if (peek.next(nx) && r < R) {
          const char* nq = reinterpret_cast<const char*>(prm.q + (static_cast<size_t>(nx.b) * R + r) * kD);
          for (int o = hf * (kD * 2 / 2); o < (hf + 1) * (kD * 2 / 2); o += 128) prefetch_l2(nq + o);
        }
      }

      // keys visible to this row (bottom-right causal alignment); pages wholly
      // below every row's limit need no mask
      const int qtok = (r < R) ? r / prm.h_q : 0;
      const int visible = prm.causal ? (sg.s_k - prm.s_q + qtok + 1) : sg.s_k;
      const int min_visible = prm.causal ? (sg.s_k - prm.s_q + 1) : sg.s_k;
      float m_run = kNegInf, l_run = 0.f;  // l_run sums the scaled p (2^kPLog2 p)
      bool ok = true;
      for (int pg = sg.lo; pg < sg.hi; ++pg, ++i) {
        if (!warp_wait(&bars->s_full, i & 1, abort_flag, __LINE__)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s[32];
        tmem_ld32(lane_base + C::kTS + 32 * hf, s);
        tmem_ld_wait();
        tc_fence_before();
        warp_arrive(&bars->s_free);

        float mx = kNegInf;
        if (pg * kPage + kPage > min_visible) {
          const int base = pg * kPage + 32 * hf;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float v = (base + c < visible) ? __uint_as_float(s[c]) : kNegInf;
            s[c] = __float_as_uint(v);
            mx = fmaxf(mx, v);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) mx = fmaxf(mx, __uint_as_float(s[c]));
        }
        mx *= c_row;  // c_row > 0
        float* xm = &bars->xmax[i & 1][0][0];
        xm[hf * kRows + r] = mx;
        if (!xsync()) {
          ok = false;
          break;
        }
        mx = fmaxf(xm[r], xm[kRows + r]);
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_run + C::kTau) {
          alpha = ex2_approx(m_run - mx);
          rescale = (pg != sg.lo);
          m_run = mx;
        }
        const float bias = (m_run == kNegInf) ? 0.f : (C::kPLog2 - m_run);
        float sum = 0.f;
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(s[c]), c_row, bias));
          const float p1 = ex2_approx(fmaf(__uint_as_float(s[c + 1]), c_row, bias));
          const float p2 = ex2_approx(fmaf(__uint_as_float(s[c + 2]), c_row, bias));
          const float p3 = ex2_approx(fmaf(__uint_as_float(s[c + 3]), c_row, bias));
          sum += (p0 + p1) + (p2 + p3);
          {
            pk[c / 2] = pack_bf16x2(p0, p1);
            pk[c / 2 + 1] = pack_bf16x2(p2, p3);
          }
        }
        l_run = l_run * alpha + sum;

        if (i > 0 && !warp_wait(&bars->pv_done, (i - 1) & 1, abort_flag, __LINE__)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
          const float f = rescale ? alpha : 1.f;
#pragma unroll 1
          for (int ch = 0; ch < kOHalf / 32; ++ch) {
            const uint32_t col = C::kTO + hf * kOHalf + ch * 32;
            uint32_t o[32];
            tmem_ld32(lane_base + col, o);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
            tmem_st32(lane_base + col, o);
          }
        }
        tmem_st16(lane_base + C::kTP + 16 * hf, pk);
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&bars->p_full);
      }
      if (!ok) break;

      // ---- epilogue: O is final once the segment's last P.V completes ----
      if (!warp_wait(&bars->pv_done, (i - 1) & 1, abort_flag, __LINE__)) break;
      tc_fence_after();
      bars->xsum[hf][r] = l_run;
      if (!xsync()) break;
      const float l_tot = (bars->xsum[0][r] + bars->xsum[1][r]) * (1.0f / C::kPScale);  // sum of p
      const bool whole = (sg.lo == 0 && sg.hi == sg.n);
      const float o_scale = kv_scale / C::kPScale;  // tensor-core units -> true units
      const float f = whole ? ((l_tot > 0.f) ? o_scale / l_tot : 0.f) : o_scale;
      const int col0 = part * C::kDvPart + hf * kOHalf;
      const int slot = whole ? 0 : prm.num_splits[sg.b] + sg.split;
#pragma unroll 1
      for (int ch = 0; ch < kOHalf / 32; ++ch) {
        uint32_t o[32];
        tmem_ld32(lane_base + C::kTO + hf * kOHalf + ch * 32, o);
        tmem_ld_wait();
        if (r >= R) continue;
        if (whole) {
          uint4* dst = reinterpret_cast<uint4*>(prm.out + (static_cast<size_t>(sg.b) * R + r) * kDV + col0 + ch * 32);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * f, __uint_as_float(o[8 * c + 1]) * f);
            w.y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * f, __uint_as_float(o[8 * c + 3]) * f);
            w.z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * f, __uint_as_float(o[8 * c + 5]) * f);
            w.w = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * f, __uint_as_float(o[8 * c + 7]) * f);
            dst[c] = w;
          }
        } else {
          uint4* dst = reinterpret_cast<uint4*>(prm.ws_o + (static_cast<size_t>(slot) * kRows + r) * kDV + col0 + ch * 32);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * f, __uint_as_float(o[8 * c + 1]) * f);
            w.y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * f, __uint_as_float(o[8 * c + 3]) * f);
            w.z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * f, __uint_as_float(o[8 * c + 5]) * f);
            w.w = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * f, __uint_as_float(o[8 * c + 7]) * f);
            dst[c] = w;
          }
        }
      }
      if (r < R && hf == 0) {
        const size_t row = static_cast<size_t>(sg.b) * R + r;
        if (whole) {
          if (part == 0) prm.lse[row] = (l_tot > 0.f) ? (m_run + lg2_approx(l_tot)) * kLn2 : kNegInf;
        } else {
          const size_t srow = static_cast<size_t>(slot) * kRows + r;
          if (part == 0) prm.ws_ml[srow] = make_float2((l_tot > 0.f) ? m_run : kNegInf, l_tot);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// FP8-dots kernel.
//
// Work unit = 2 CTAs, each owning one 256-wide dv slice [256 part, +256).
// Both walk the unit's pages two at a time: block h is pages 2i and 2i + 1 of
// a segment, or its last page alone.  Each CTA computes the block's scores
// S = Q K^T as one 128-row x 128-key tile and its probabilities P itself (the
// two CTAs of a unit compute the same S and P; a tcgen05 MMA with M = 128
// costs nearly the same for any N up to 256, so the 128-key tiles take half
// the tensor time per key of 64-key ones), then multiplies P by its dv slice
// of the block's V.
//
// TMEM: O slice (256 columns), S (128), Q latent (128, E4M3).  Shared memory:
// a V ring with this CTA's latent half of each block (3 x 32 KB, released by
// the block's P.V; Q.K^T reads it too), a ring of five 16 KB K slices (per
// block three: the other latent half's two 128-byte boxes, then the RoPE
// part, converted to f16 in place; each released when its Q.K^T step
// completes; five keep the next block's slices and part of the one after in
// flight, since a slice takes over a microsecond to land),
// Q's RoPE part (f16), P (128 rows x 128 E4M3 keys) and the unit's first
// block-table entries.
// ===========================================================================
namespace f8 {
constexpr int kThreads = 384;
constexpr int kBlkPages = 2;
constexpr int kBlkKeys = kBlkPages * kPage;   // keys of a full block (N of its Q.K^T)
constexpr int kVStages = 3;
constexpr int kKSlices = 5;
constexpr int kBoxBlk = kBlkPages * kLatBox;  // one 128-byte column box of a block: page 0 rows, then page 1 rows
constexpr int kVBytes = 2 * kBoxBlk;          // latent bytes [256 part, 256 part + 256) of a block
constexpr int kSliceBytes = kBoxBlk;
constexpr int kRopeRaw = kPage * 64;          // in a page's 8 KB of a RoPE slice: where its E4M3 bytes land
constexpr int kOffV = 0;
constexpr int kOffK = kOffV + kVStages * kVBytes;
constexpr int kOffQRope = kOffK + kKSlices * kSliceBytes;  // Q RoPE, 128 rows x 64 f16, 128-byte swizzle
constexpr int kOffP = kOffQRope + kRows * 128;
constexpr int kPBytes = kRows * kBlkKeys;  // P: 128 rows x 128 E4M3 keys
constexpr int kOffPtab = kOffP + kPBytes;  // the unit's first kPtabMax block-table entries
constexpr int kPtabMax = 2048;
constexpr int kSmemData = kOffPtab + kPtabMax * 4;
// P: 8-row x 16-byte core matrices, key chunk c of row group G at c * kPLbo + G * kPSbo, so the 32
// rows x 16 bytes that one warp writes per key chunk are one contiguous 512-byte piece
constexpr int kPLbo = 2048, kPSbo = 128;
constexpr float kPScale = 64.0f, kPLog2 = 6.0f;  // P is stored as E4M3(64 p)
constexpr float kTau = 2.75f;                    // 64 * 2^2.75 = 430.5 < 448
// TMEM columns: O slice, S, Q latent (E4M3, the A operand of the latent Q.K^T)
constexpr uint32_t kTO = 0, kTS = 256, kTQ = 384;
static_assert(kVBytes % 1024 == 0 && kOffK % 1024 == 0 && kSliceBytes % 1024 == 0 && kOffQRope % 1024 == 0 &&
                  kOffP % 1024 == 0,
              "1 KB aligned tiles");
// Quantised Q of a sequence (written by mla_qprep_kernel): per row latent bytes
// [256 h, 256 h + 256) at a 272-byte pitch for h = 0, 1, then the RoPE values as
// f16 at a 144-byte pitch (pitches chosen so a quarter-warp's 16-byte row
// accesses hit distinct banks).
constexpr int kQLatPitch = 272;
constexpr int kQRopePitch = 144;
constexpr int kQLatSlotBytes = kRows * kQLatPitch;
constexpr int kQRopeSlotBytes = kRows * kQRopePitch;
// After the slots: the latent quantisation error q_hat qs - q, 128 rows x 512
// bf16, read by the combine kernel for the LSE correction.
constexpr int kQErrOff = 2 * kQLatSlotBytes + kQRopeSlotBytes;
static_assert(kQErrOff == kMlaQErrOff && kQErrOff + kRows * kDLat * 2 == kMlaQBytes, "quantised-Q layout");

struct Bars {
  uint64_t v_full[kVStages];   // by block h % kVStages: this CTA's latent half of block h loaded
  uint64_t v_empty[kVStages];  // its P.V (after its Q.K^T) completed
  uint64_t k_full[kKSlices];   // by slice n % kKSlices (slices 3h, 3h + 1, 3h + 2 of block h) loaded
  uint64_t k_empty[kKSlices];  // the slice's Q.K^T step completed
  uint64_t k_cvt[2];           // by block h % 2: its RoPE slice converted to f16
  uint64_t s_full;             // S holds block h's scores
  uint64_t s_free;             // S read out (8 softmax warps)
  uint64_t p_full;             // P written and O rescaled (8 softmax warps)
  uint64_t pv_done;            // the block's P.V completed
  uint64_t rmax_full[4];       // by row group: both halves' row maxima written (2 warps)
  uint64_t q_full;             // a segment's Q copied in (8 softmax warps)
  uint64_t ptab_ready;         // the block-table entries are in shared memory
  uint64_t final_mma, xchg;
  uint32_t tmem_base, abort_flag, cvt_ok;
  float xsum[2][2][kRows];  // by segment parity: row-sum halves of the two softmax threads of a row
  float rmax[2][2][kRows];  // by block parity: the row maxima of the two halves of a row
};
static_assert(kSmemData % 16 == 0, "the barrier block starts 16-byte aligned");

constexpr size_t smem_bytes() { return kSmemData + sizeof(Bars) + 1024; }
static_assert(smem_bytes() <= 232448, "fits the 227 KB opt-in shared memory of a CTA");

// Test hook of the bounded waits (0 = off); set by mla_set_wait_test.
__device__ int g_fault_page = 0;

// Blocks of a unit one at a time: h counts the unit's blocks across
// segments, seg its non-empty segments; the block is pages [pg, pg + npg),
// and u0 + (pg - sg.lo) is the unit's page count before it.
struct BlockCursor {
  SegmentWalker walk;
  Segment sg;
  int pg = 0, npg = 0, h = -1, seg = -1, u0 = 0;
  bool valid = false;
  __device__ BlockCursor(const MlaParams& p, int unit) : walk(p, unit) {}
  __device__ bool next() {
    if (valid && pg + npg < sg.hi) {
      pg += npg;
    } else {
      if (valid) u0 += sg.hi - sg.lo;
      valid = walk.next(sg);
      if (!valid) return false;
      pg = sg.lo;
      ++seg;
    }
    npg = min(kBlkPages, sg.hi - pg);
    ++h;
    return true;
  }
  __device__ bool first() const { return pg == sg.lo; }
  __device__ bool last() const { return pg + npg == sg.hi; }
  __device__ int upage() const { return u0 + (pg - sg.lo); }
};

// Quantises the Q rows of sequence b into the three Q slots: latent -> E4M3(q / qs),
// RoPE -> f16(q / qs), qs = smallest power of two with amax <= 448 qs.  kTpr
// threads share a row; thread `part` takes the 8-value chunks c = part (mod kTpr)
// of the row's 72 (64 latent, 8 RoPE).
template <int kTpr>
__device__ __forceinline__ void fill_q_row(const MlaParams& prm, int b, int r, int part, uint8_t* slot0,
                                           uint8_t* slot1, uint8_t* slot2, uint8_t* err, float* qs_out) {
  constexpr int kChunks = 72 / kTpr;
  constexpr bool kHold = kChunks <= 18;  // few enough chunks to keep in registers between the two passes
  const int R = prm.s_q * prm.h_q;
  const bool live = r < R;
  const uint4* q4 = reinterpret_cast<const uint4*>(prm.q + (static_cast<size_t>(b) * R + (live ? r : 0)) * kD);
  uint4 held[kHold ? kChunks : 1];
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < kChunks; ++j) {
    const uint4 v = live ? __ldg(q4 + part + j * kTpr) : make_uint4(0, 0, 0, 0);
    if constexpr (kHold) held[j] = v;
    amax = fmaxf(amax, absmax_bf16x8(v));
  }
#pragma unroll
  for (int o = 1; o < kTpr; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int qe = pow2_scale_exponent(amax);
  const float inv_qs = exp2i(-qe);
  // chunk c (8 values) -> latent bytes of slot c / 32, or f16 RoPE of slot 2
  auto put = [&](int c, uint4 a) {
    if (c < 64) {
      uint2 o;
      o.x = pack_e4m3x4(bf16_lo(a.x) * inv_qs, bf16_hi(a.x) * inv_qs, bf16_lo(a.y) * inv_qs, bf16_hi(a.y) * inv_qs);
      o.y = pack_e4m3x4(bf16_lo(a.z) * inv_qs, bf16_hi(a.z) * inv_qs, bf16_lo(a.w) * inv_qs, bf16_hi(a.w) * inv_qs);
      uint8_t* slot = (c < 32) ? slot0 : slot1;
      *reinterpret_cast<uint2*>(slot + r * kQLatPitch + (c & 31) * 8) = o;
      const float qs = exp2i(qe);
      const uint32_t w[4] = {a.x, a.y, a.z, a.w};
      const uint32_t hq[4] = {e4m3x2_to_f16x2(o.x & 0xFFFFu), e4m3x2_to_f16x2(o.x >> 16), e4m3x2_to_f16x2(o.y & 0xFFFFu),
                              e4m3x2_to_f16x2(o.y >> 16)};
      uint4 ev;
      uint32_t* e4 = &ev.x;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        e4[k] = pack_bf16x2(f16_lo(hq[k]) * qs - bf16_lo(w[k]), f16_hi(hq[k]) * qs - bf16_hi(w[k]));
      *reinterpret_cast<uint4*>(err + r * kDLat * 2 + c * 16) = ev;
    } else {
      uint4 o;
      o.x = pack_f16x2(bf16_lo(a.x) * inv_qs, bf16_hi(a.x) * inv_qs);
      o.y = pack_f16x2(bf16_lo(a.y) * inv_qs, bf16_hi(a.y) * inv_qs);
      o.z = pack_f16x2(bf16_lo(a.z) * inv_qs, bf16_hi(a.z) * inv_qs);
      o.w = pack_f16x2(bf16_lo(a.w) * inv_qs, bf16_hi(a.w) * inv_qs);
      *reinterpret_cast<uint4*>(slot2 + r * kQRopePitch + (c - 64) * 16) = o;
    }
  };
  if constexpr (kHold) {
#pragma unroll
    for (int j = 0; j < kChunks; ++j) put(part + j * kTpr, held[j]);
  } else {
#pragma unroll 6
    for (int j = 0; j < kChunks; ++j) {
      const int c = part + j * kTpr;
      put(c, live ? __ldg(q4 + c) : make_uint4(0, 0, 0, 0));
    }
  }
  if (part == 0) qs_out[r] = exp2i(qe);
}
// Quantised Q for FP8 dots in the ring's Q-slot layout, one grid ahead of the
// decode kernel: grid (b, 4), 256 threads, eight threads per row, 32 rows per
// CTA.  It is the first kernel of a decode call and is launched as a
// programmatic dependent of whatever the caller enqueued before (which may
// have written Q), so it waits for that work before reading Q; it lets the
// decode kernel start its prologue at once, and the decode kernel's wait on
// this grid then also covers the tile schedule written before it.
__global__ void __launch_bounds__(256) mla_qprep_kernel(const MlaParams prm) {
  griddep_launch_dependents();
  griddep_wait();
  const int b = blockIdx.x;
  const int r = blockIdx.y * 32 + threadIdx.x / 8;
  uint8_t* q = prm.qbuf + static_cast<size_t>(b) * kMlaQBytes;
  fill_q_row<8>(prm, b, r, threadIdx.x % 8, q, q + kQLatSlotBytes, q + 2 * kQLatSlotBytes, q + kQErrOff,
                prm.qscale + static_cast<size_t>(b) * kRows);
}

// Lanes in groups of N (N = 4 or 8) each hold N 16-byte pieces; afterwards
// lane q of a group holds piece q of every lane of its group, piece k coming
// from lane k (an N x N transpose by XOR butterflies).
template <int N>
__device__ __forceinline__ void lane_group_transpose(uint4 (&pc)[N], int lane) {
  const int q = lane & (N - 1);
#pragma unroll
  for (int m = N / 2; m >= 1; m >>= 1) {
    const bool hi = (q & m) != 0;
#pragma unroll
    for (int a = 0; a < N; ++a) {
      if (a & m) continue;
      const int b = a | m;
      uint4 t = hi ? pc[a] : pc[b];  // the piece the partner needs
      t.x = __shfl_xor_sync(0xffffffffu, t.x, m);
      t.y = __shfl_xor_sync(0xffffffffu, t.y, m);
      t.z = __shfl_xor_sync(0xffffffffu, t.z, m);
      t.w = __shfl_xor_sync(0xffffffffu, t.w, m);
      if (hi)
        pc[a] = t;
      else
        pc[b] = t;
    }
  }
}
}  // namespace f8

__global__ void __launch_bounds__(f8::kThreads, 1)
    mla_fp8_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope,
                   const MlaParams prm) {
  using namespace f8;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + kSmemData);
  volatile uint32_t* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int unit = blockIdx.x / 2;
  const int part = blockIdx.x % 2;  // dv slice [256 part, 256 part + 256); this CTA's latent half
  const int other = part ^ 1;       // the other latent half (Q.K^T only)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int s = 0; s < kKSlices; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&bars->k_cvt[b], 1);
    for (int b = 0; b < 4; ++b) mbar_init(&bars->rmax_full[b], 2);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, kSoftmaxThreads / 32);
    mbar_init(&bars->p_full, kSoftmaxThreads / 32);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->q_full, kSoftmaxThreads / 32);
    mbar_init(&bars->ptab_ready, 1);
    mbar_init(&bars->final_mma, 1);
    mbar_init(&bars->xchg, kSoftmaxThreads / 32);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  // Everything above overlaps the previous kernel (launched as its dependent);
  // from here on this grid reads the schedule and the quantised Q.
  griddep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer ----
    // Two streams of loads, issued by lane 0 as their stages free up: the V
    // half of every block (this CTA's latent bytes [256 part, +256) of each
    // page) and the three K slices of every block (the other latent half's
    // two boxes, then the RoPE bytes).
    if (lane == 0) {
      tma_prefetch_desc(&tm_lat);
      tma_prefetch_desc(&tm_rope);
      // bounded-wait test hook: CTA 0 of unit 0 never loads the block holding its page g_fault_page - 1
      const int fault = (unit == 0 && part == 0) ? *reinterpret_cast<volatile int*>(&g_fault_page) : 0;
      auto skipped = [&](const BlockCursor& c) { return fault > c.upage() && fault <= c.upage() + c.npg; };
      const int32_t* ptab = reinterpret_cast<const int32_t*>(smem + kOffPtab);
      bool ptab_ok = false;
      // a block-table entry: from the shared-memory copy once it is in, else from global memory
      auto phys_of = [&](const BlockCursor& c, int i) -> int {
        const int u = c.upage() + i;
        if (!ptab_ok && u < kPtabMax) ptab_ok = mbar_test_wait(&bars->ptab_ready, 0);
        int ph = (ptab_ok && u < kPtabMax)
                     ? ptab[u]
                     : __ldg(prm.block_table + static_cast<size_t>(c.sg.b) * prm.max_pages + c.pg + i);
        if (ph < 0 || ph >= prm.num_pages) {
          atomicOr(&g_status_mla, FP8MLA_DEV_BAD_PAGE);
          ph = 0;
        }
        return ph;
      };
      BlockCursor vc(prm, unit), kc(prm, unit);  // next block to load V for; next block for K slices
      bool v_more = vc.next(), k_more = kc.next();
      int vp0 = 0, vp1 = 0, kp0 = 0, kp1 = 0;  // physical pages of those blocks
      if (v_more) {
        vp0 = phys_of(vc, 0);
        vp1 = vc.npg > 1 ? phys_of(vc, 1) : 0;
      }
      if (k_more) {
        kp0 = phys_of(kc, 0);
        kp1 = kc.npg > 1 ? phys_of(kc, 1) : 0;
      }
      int kn = 0, ks = 0;  // K slices issued; slice of the current block (0, 1 latent, 2 RoPE)
      uint32_t v_last = 0, v_par = 0, k_last = 0, k_par = 0;  // per stage: loaded here, and its phase parity
      uint32_t polls = 0;
      uint64_t t_idle = 0;
      bool ok = true;
      while (ok && (v_more || k_more)) {
        bool did = false;
        if (k_more) {
          const int st = kn % kKSlices, use = kn / kKSlices;
          if (use == 0 || mbar_test_wait(&bars->k_empty[st], (use - 1) & 1)) {
            if (!skipped(kc)) {
              uint8_t* sb = smem + kOffK + st * kSliceBytes;
              mbar_arrive_expect_tx(&bars->k_full[st], static_cast<uint32_t>((ks < 2 ? kLatBox : kRopeRaw) * kc.npg));
              if (ks < 2) {
                tma_load_3d(sb, &tm_lat, &bars->k_full[st], other * 256 + ks * 128, 0, kp0);
                if (kc.npg > 1) tma_load_3d(sb + kLatBox, &tm_lat, &bars->k_full[st], other * 256 + ks * 128, 0, kp1);
              } else {
                tma_load_3d(sb + kRopeRaw, &tm_rope, &bars->k_full[st], kDLat, 0, kp0);
                if (kc.npg > 1) tma_load_3d(sb + kLatBox + kRopeRaw, &tm_rope, &bars->k_full[st], kDLat, 0, kp1);
              }
              k_last |= 1u << st;
              k_par = (k_par & ~(1u << st)) | (static_cast<uint32_t>(use & 1) << st);
            }
            ++kn;
            if (++ks == 3) {
              ks = 0;
              k_more = kc.next();
              if (k_more) {
                kp0 = phys_of(kc, 0);
                kp1 = kc.npg > 1 ? phys_of(kc, 1) : 0;
              }
            }
            did = true;
          }
        }
        if (v_more && (vc.h < kVStages ||
                       mbar_test_wait(&bars->v_empty[vc.h % kVStages], ((vc.h / kVStages) - 1) & 1))) {
          const int st = vc.h % kVStages;
          if (!skipped(vc)) {
            uint8_t* sb = smem + kOffV + st * kVBytes;
            mbar_arrive_expect_tx(&bars->v_full[st], static_cast<uint32_t>(2 * kLatBox * vc.npg));
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              tma_load_3d(sb + q * kBoxBlk, &tm_lat, &bars->v_full[st], part * 256 + q * 128, 0, vp0);
              if (vc.npg > 1)
                tma_load_3d(sb + q * kBoxBlk + kLatBox, &tm_lat, &bars->v_full[st], part * 256 + q * 128, 0, vp1);
            }
            v_last |= 1u << st;
            v_par = (v_par & ~(1u << st)) | (static_cast<uint32_t>((vc.h / kVStages) & 1) << st);
          }
          v_more = vc.next();
          if (v_more) {
            vp0 = phys_of(vc, 0);
            vp1 = vc.npg > 1 ? phys_of(vc, 1) : 0;
          }
          did = true;
        }
        if (did) {
          polls = 0;
        } else if ((++polls & 255u) == 0) {
          if (*abort_flag) ok = false;
          if (polls == 256) t_idle = globaltimer_ns();
          if (ok && polls > kWaitMinPolls && globaltimer_ns() - t_idle > *(volatile uint64_t*)&g_wait_limit_ns) {
            atomicOr(&g_status_mla, FP8MLA_DEV_WAIT_TIMEOUT);
            record_timeout_site(__LINE__);
            ok = false;
          }
        }
      }
      if (!ok) *abort_flag = 1u;
      // Never leave with copies in flight: wait for the last load of each stage.
      for (int st = 0; st < kKSlices; ++st)
        if ((k_last >> st) & 1u) wait_bounded(&bars->k_full[st], (k_par >> st) & 1u, nullptr, &g_status_mla, __LINE__);
      for (int st = 0; st < kVStages; ++st)
        if ((v_last >> st) & 1u) wait_bounded(&bars->v_full[st], (v_par >> st) & 1u, nullptr, &g_status_mla, __LINE__);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer ----
    // The whole warp runs the loop and one elected lane issues.  The warp
    // polls the next block's P.V and the next step of the next block's Q.K^T
    // and issues whichever is ready (P.V first: it frees a V stage and P), so
    // neither waits behind the other.  Q.K^T(h) runs in four steps: this
    // CTA's latent half from the V stage once S is read out and, when the
    // block opens a segment, that segment's Q is in (the stage is probed only
    // after the P.V of its previous block was issued, so the probe cannot see
    // that block's phase); the other latent half's two boxes (K slices); and
    // the converted RoPE slice.  P.V(h) needs P(h) written and O rescaled.
    // Before the P.V of a block holding a sequence's last page the warp zeroes
    // that page's V rows past the sequence end (they may hold anything, and P
    // is 0 there).
    constexpr uint32_t idesc_pv = make_idesc(0, 0, 0, 1, 256, 128);  // e4m3, B MN-major, N = 256
    const bool leader = elect_one();
    const uint64_t qd = make_sdesc(smem_u32(smem + kOffQRope), 16, 1024, SWIZZLE_128B);
    const uint64_t pd = make_sdesc(smem_u32(smem + kOffP), kPLbo, kPSbo, SWIZZLE_NONE);
    BlockCursor qk(prm, unit);  // next block whose Q.K^T is due
    BlockCursor pv(prm, unit);  // next block whose P.V is due
    int qn = 0, qk_seg = -1, step = 0;  // Q copies consumed, segment of the last Q.K^T, next step
    bool qk_more = qk.next();
    bool pv_more = pv.next();
    bool ok = true;
    uint64_t t_idle = 0;
    uint32_t polls = 0;
    while (ok && (qk_more || pv_more)) {
      bool did = false;
      if (pv_more) {
        const int h = pv.h;
        const int st = h % kVStages;
        const bool ready = mbar_test_wait(&bars->p_full, h & 1) && mbar_test_wait(&bars->v_full[st], (h / kVStages) & 1);
        if (__all_sync(0xffffffffu, ready)) {
          uint8_t* vs = smem + kOffV + st * kVBytes;
          if (pv.pg + pv.npg == pv.sg.n) {  // the sequence's last page: zero its rows past the end
            const int lp = pv.npg - 1;
            const int live = pv.sg.s_k - (pv.pg + lp) * kPage;  // rows of the page that hold keys
            if (live < kPage) {
              const uint4 z = make_uint4(0, 0, 0, 0);
              for (int i = lane; i < (kPage - live) * 16; i += 32) {
                const int row = live + i / 16, c = i % 16;
                *reinterpret_cast<uint4*>(vs + (c >> 3) * kBoxBlk + lp * kLatBox + row * 128 + ((c & 7) << 4)) = z;
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
          }
          tc_fence_after();
          const uint64_t vd = make_sdesc(smem_u32(vs), kBoxBlk, 1024, SWIZZLE_128B);
          const bool first = pv.first();
          for (int kk = 0; kk < 2 * pv.npg; ++kk)
            mma_f8_ss_if(leader, tmem + kTO, pd + ((kk * 2 * kPLbo) >> 4), vd + ((kk * 4096) >> 4), idesc_pv,
                         (first && kk == 0) ? 0u : 1u);
          tc_commit_if(leader, &bars->pv_done);
          tc_commit_if(leader, &bars->v_empty[st]);
          pv_more = pv.next();
          did = true;
        }
      }
      if (!did && qk_more) {
        const int h = qk.h;
        const uint32_t n_keys = static_cast<uint32_t>(kPage * qk.npg);
        const uint32_t idesc8 = make_idesc(0, 0, 0, 0, n_keys, 128);   // e4m3 x e4m3, both K-major
        const uint32_t idesc16 = make_idesc(0, 0, 0, 0, n_keys, 128);  // f16 x f16 (E4M3 keys are exact in f16)
        if (step == 0) {
          const bool opens = qk.seg != qk_seg;
          const int vst = h % kVStages;
          const bool ready = (!opens || mbar_test_wait(&bars->q_full, qn & 1)) &&
                             (h < 1 || mbar_test_wait(&bars->s_free, (h - 1) & 1)) &&
                             (!pv_more || pv.h > h - kVStages) &&
                             mbar_test_wait(&bars->v_full[vst], (h / kVStages) & 1);
          if (__all_sync(0xffffffffu, ready)) {
            if (opens) {
              qk_seg = qk.seg;
              ++qn;
            }
            tc_fence_after();
            const uint64_t vd = make_sdesc(smem_u32(smem + kOffV + vst * kVBytes), 16, 1024, SWIZZLE_128B);
            // boxes q = 2 part + i hold Q.K^T bytes [128 q, 128 q + 128) of the keys
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f8_ts_if(leader, tmem + kTS, tmem + kTQ + (4 * (2 * part + i) + kk) * 8,
                             vd + ((i * kBoxBlk + kk * 32) >> 4), idesc8, (i | kk) ? 1u : 0u);
            step = 1;
            did = true;
          }
        } else {
          const int n = 3 * h + step - 1;  // steps 1, 2: the other latent boxes; step 3: RoPE
          const int st = n % kKSlices;
          const bool ready = step < 3 ? mbar_test_wait(&bars->k_full[st], (n / kKSlices) & 1)
                                      : mbar_test_wait(&bars->k_cvt[h & 1], (h >> 1) & 1);
          if (__all_sync(0xffffffffu, ready)) {
            tc_fence_after();
            const uint64_t kd = make_sdesc(smem_u32(smem + kOffK + st * kSliceBytes), 16, 1024, SWIZZLE_128B);
            if (step < 3) {
              const int q = 2 * other + step - 1;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f8_ts_if(leader, tmem + kTS, tmem + kTQ + (4 * q + kk) * 8, kd + ((kk * 32) >> 4), idesc8, 1u);
            } else {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f16_ss_if(leader, tmem + kTS, qd + ((kk * 32) >> 4), kd + ((kk * 32) >> 4), idesc16, 1u);
            }
            tc_commit_if(leader, &bars->k_empty[st]);
            if (step == 3) {
              tc_commit_if(leader, &bars->s_full);
              step = 0;
              qk_more = qk.next();
            } else {
              ++step;
            }
            did = true;
          }
        }
      }
      // bounded: no progress for the wait limit (or another role stopped) ends the loop
      if (did) {
        polls = 0;
      } else if ((++polls & 255u) == 0) {
        if (*abort_flag) ok = false;
        if (polls == 256) t_idle = globaltimer_ns();
        if (ok && polls > kWaitMinPolls && globaltimer_ns() - t_idle > *(volatile uint64_t*)&g_wait_limit_ns) {
          if (lane == 0) {
            atomicOr(&g_status_mla, FP8MLA_DEV_WAIT_TIMEOUT);
            record_timeout_site(__LINE__);
          }
          ok = false;
        }
        ok = __all_sync(0xffffffffu, ok);
      }
    }
    if (!ok && lane == 0) *abort_flag = 1u;
    if (leader) tc_commit(&bars->final_mma);
    __syncwarp();
    warp_wait(&bars->final_mma, 0, nullptr, __LINE__);
  } else if (warp == 2 || warp == 3) {
    // ---------------------- RoPE conversion (64 threads) ----
    // First the unit's block-table entries (as many as fit) go into shared
    // memory for the producer.  Then thread 0 waits for every K slice in order
    // (so no wait can see a stage's phase two ahead), and for a block's RoPE
    // slice thread t reads the E4M3 RoPE bytes of token row t of each page
    // from the second half of the page's 8 KB and, after all have read, writes
    // them as f16 (exact) over the whole 8 KB, 128-byte swizzled; rows past
    // the sequence end become 0 (their scores are masked anyway).
    const int t = threadIdx.x - 64;  // token row of a page
    {
      int32_t* ptab = reinterpret_cast<int32_t*>(smem + kOffPtab);
      SegmentWalker w(prm, unit);
      Segment sg;
      int u0 = 0;
      while (u0 < kPtabMax && w.next(sg)) {
        const int32_t* row = prm.block_table + static_cast<size_t>(sg.b) * prm.max_pages;
        const int n = min(sg.hi - sg.lo, kPtabMax - u0);
        for (int i = t; i < n; i += 64) cp_async4(ptab + u0 + i, row + sg.lo + i);
        u0 += n;
      }
      cp_async_wait_all();
      named_bar_sync(1, 64);
      if (t == 0) mbar_arrive(&bars->ptab_ready);
    }
    BlockCursor bc(prm, unit);
    bool ok = true;
    int n = 0;  // K slices waited for
    while (ok && bc.next()) {
      const int st = (n + 2) % kKSlices;
      if (t == 0) {
        bool good = true;
        for (int s3 = 0; s3 < 3 && good; ++s3)
          good = wait_bounded(&bars->k_full[(n + s3) % kKSlices], ((n + s3) / kKSlices) & 1, abort_flag,
                              &g_status_mla, __LINE__);
        bars->cvt_ok = good ? 1u : 0u;
      }
      n += 3;
      named_bar_sync(1, 64);
      if (!bars->cvt_ok) {
        ok = false;
        break;
      }
      uint8_t* kb = smem + kOffK + st * kSliceBytes;
      const uint4 z = make_uint4(0, 0, 0, 0);
      uint4 raw[kBlkPages][4];
#pragma unroll
      for (int i = 0; i < kBlkPages; ++i) {
        const bool dead = i >= bc.npg || (bc.pg + i == bc.sg.n - 1 && t >= bc.sg.s_k - (bc.pg + i) * kPage);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          raw[i][c] = dead ? z : reinterpret_cast<const uint4*>(kb + i * kLatBox + kRopeRaw + t * 64)[c];
      }
      named_bar_sync(1, 64);  // every raw row is read before the f16 rows overwrite them
      const int sw = t & 7;
#pragma unroll
      for (int i = 0; i < kBlkPages; ++i) {
        if (i >= bc.npg) break;
        uint8_t* dst = kb + i * kLatBox + t * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = raw[i][c];
          uint4 lo, hi;
          lo.x = e4m3x2_to_f16x2(v.x & 0xFFFFu);
          lo.y = e4m3x2_to_f16x2(v.x >> 16);
          lo.z = e4m3x2_to_f16x2(v.y & 0xFFFFu);
          lo.w = e4m3x2_to_f16x2(v.y >> 16);
          hi.x = e4m3x2_to_f16x2(v.z & 0xFFFFu);
          hi.y = e4m3x2_to_f16x2(v.z >> 16);
          hi.z = e4m3x2_to_f16x2(v.w & 0xFFFFu);
          hi.w = e4m3x2_to_f16x2(v.w >> 16);
          *reinterpret_cast<uint4*>(dst + (((2 * c) ^ sw) << 4)) = lo;
          *reinterpret_cast<uint4*>(dst + (((2 * c + 1) ^ sw) << 4)) = hi;
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 64);
      if (t == 0) mbar_arrive(&bars->k_cvt[bc.h & 1]);
    }
    if (!ok && t == 0) *abort_flag = 1u;
  } else {
    // ------------------ softmax / Q copy / epilogue (8 warps, 2 per row) ----
    const int hf = (warp - 4) / 4;         // which half of the row (keys [64 hf, 64 hf + 64) of a block)
    const int r = (warp % 4) * 32 + lane;  // query row = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    const float kv_scale = *prm.kv_scale;
    const int R = prm.s_q * prm.h_q;
    constexpr int kOHalf = 128;  // O columns of this thread
    uint32_t xphase = 0;
    auto xsync = [&]() -> bool {  // bounded, abort-aware exchange point of the 256 softmax threads
      warp_arrive(&bars->xchg);
      const bool ok = warp_wait(&bars->xchg, xphase & 1, abort_flag, __LINE__);
      ++xphase;
      return ok;
    };
    const uint32_t prow = static_cast<uint32_t>((r >> 3) * kPSbo + (r & 7) * 16);

    // Copies this half of sequence b_seq's quantised Q row (prepared by
    // mla_qprep_kernel) in: latent bytes [256 hf, +256) into TMEM columns
    // kTQ + 64 hf.., RoPE values [32 hf, +32) into the Q RoPE tile.
    float qs_cur = 1.f;
    auto copy_q = [&](int b_seq) {
      const uint8_t* qb = prm.qbuf + static_cast<size_t>(b_seq) * kMlaQBytes;
      const uint4* lat = reinterpret_cast<const uint4*>(qb + hf * kQLatSlotBytes + r * kQLatPitch);
      const uint4* rope = reinterpret_cast<const uint4*>(qb + 2 * kQLatSlotBytes + r * kQRopePitch + hf * 64);
      uint4 v[16], w[4];
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] = __ldg(lat + c);
#pragma unroll
      for (int c = 0; c < 4; ++c) w[c] = __ldg(rope + c);
      qs_cur = __ldg(prm.qscale + static_cast<size_t>(b_seq) * kRows + r);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          pk[4 * c + 0] = v[4 * ch + c].x;
          pk[4 * c + 1] = v[4 * ch + c].y;
          pk[4 * c + 2] = v[4 * ch + c].z;
          pk[4 * c + 3] = v[4 * ch + c].w;
        }
        tmem_st16(lane_base + kTQ + (4 * hf + ch) * 16, pk);
      }
      uint8_t* dst = smem + kOffQRope + r * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(dst + (((4 * hf + c) ^ (r & 7)) << 4)) = w[c];
      fence_proxy_async_smem();  // the Q RoPE tile is read by the MMAs
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(&bars->q_full);
    };

    BlockCursor pc(prm, unit);
    bool ok = true;
    int cur_seg = -1;
    float m_run = kNegInf, l_run = 0.f;  // reference of O and l; this thread's share of l
    int qtok = 0, visible = 0;
    float c_row = 0.f;

    // Moves O and l to a new reference before a block's P.V (whose P was
    // taken against it), once the P.V of the block before completed (the
    // caller has waited for it).
    auto rescale_to = [&](float m_new, bool first) {
      const bool rescale = !first && m_new != m_run;
      const float alpha = rescale ? ex2_approx(m_run - m_new) : 1.f;
      l_run = first ? 0.f : l_run * alpha;
      if (first || rescale) m_run = m_new;
      if (__any_sync(0xffffffffu, rescale)) {
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < kOHalf / 32; ++ch) {
          const uint32_t col = kTO + hf * kOHalf + ch * 32;
          uint32_t o[32];
          tmem_ld32(lane_base + col, o);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st32(lane_base + col, o);
        }
        tmem_st_wait();
      }
    };

    if (pc.next()) copy_q(pc.sg.b);
    pc = BlockCursor(prm, unit);

    while (ok && pc.next()) {
      const int h = pc.h;
      if (pc.seg != cur_seg) {  // a new segment
        cur_seg = pc.seg;
        m_run = kNegInf;
        l_run = 0.f;
        qtok = (r < R) ? r / prm.h_q : 0;
        visible = prm.causal ? (pc.sg.s_k - prm.s_q + qtok + 1) : pc.sg.s_k;
        c_row = prm.softmax_scale * kLog2e * qs_cur * kv_scale;
        if (r < R) {  // warm L2 with the Q of the segment after this one
          SegmentWalker peek = pc.walk;
          Segment nx;
          if (peek.next(nx)) {
            const char* nq = reinterpret_cast<const char*>(prm.qbuf + static_cast<size_t>(nx.b) * kMlaQBytes);
            prefetch_l2(nq + hf * kQLatSlotBytes + r * kQLatPitch);
            prefetch_l2(nq + hf * kQLatSlotBytes + r * kQLatPitch + 128);
          }
        }
      }
      if (!warp_spin(&bars->s_full, h & 1, abort_flag, __LINE__)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s[32], s2[32];  // keys [64 hf, +32) and [64 hf + 32, +32) of the block
      tmem_ld32(lane_base + kTS + 64 * hf, s);
      tmem_ld32(lane_base + kTS + 64 * hf + 32, s2);
      tmem_ld_wait();
      tc_fence_before();
      warp_arrive(&bars->s_free);  // block h + 1's Q.K^T may overwrite S
      // the segment's last block: its Q.K^T is done, so the next segment's Q may replace this one's
      if (pc.last()) {
        SegmentWalker peek = pc.walk;
        Segment nx;
        if (peek.next(nx)) copy_q(nx.b);
      }
      // keys past the row's causal limit or past the segment's pages
      const int key0 = pc.pg * kPage + 64 * hf;
      const int lim = min(visible, (pc.pg + pc.npg) * kPage);
      if (key0 + 64 > lim) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (key0 + c >= lim) s[c] = __float_as_uint(kNegInf);
          if (key0 + 32 + c >= lim) s2[c] = __float_as_uint(kNegInf);
        }
      }
      float m22[22];
#pragma unroll
      for (int c = 0; c < 10; ++c) {
        m22[c] = fmax3(__uint_as_float(s[3 * c]), __uint_as_float(s[3 * c + 1]), __uint_as_float(s[3 * c + 2]));
        m22[10 + c] = fmax3(__uint_as_float(s2[3 * c]), __uint_as_float(s2[3 * c + 1]), __uint_as_float(s2[3 * c + 2]));
      }
      m22[20] = fmaxf(__uint_as_float(s[30]), __uint_as_float(s[31]));
      m22[21] = fmaxf(__uint_as_float(s2[30]), __uint_as_float(s2[31]));
      float m8[8];
#pragma unroll
      for (int c = 0; c < 7; ++c) m8[c] = fmax3(m22[3 * c], m22[3 * c + 1], m22[3 * c + 2]);
      m8[7] = m22[21];
      const float mhalf = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * c_row;
      // the row's maximum: this half's, and the other half's from its thread (warp warp +- 4)
      bars->rmax[h & 1][hf][r] = mhalf;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->rmax_full[warp % 4]);
      if (!warp_spin(&bars->rmax_full[warp % 4], h & 1, abort_flag, __LINE__)) {
        ok = false;
        break;
      }
      const float mx = fmaxf(mhalf, bars->rmax[h & 1][1 - hf][r]);
      // the reference: kept unless this block's maximum exceeds it by more than kTau
      const bool first = pc.first();
      const float m_new = (first || mx > m_run + kTau) ? mx : m_run;
      const float bias = (m_new == kNegInf) ? 0.f : (kPLog2 - m_new);
      float sum = 0.f;
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(s[c]), c_row, bias));
        const float p1 = ex2_approx(fmaf(__uint_as_float(s[c + 1]), c_row, bias));
        const float p2 = ex2_approx(fmaf(__uint_as_float(s[c + 2]), c_row, bias));
        const float p3 = ex2_approx(fmaf(__uint_as_float(s[c + 3]), c_row, bias));
        sum += (p0 + p1) + (p2 + p3);
        pk[c / 4] = pack_e4m3x4(p0, p1, p2, p3);
      }
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(s2[c]), c_row, bias));
        const float p1 = ex2_approx(fmaf(__uint_as_float(s2[c + 1]), c_row, bias));
        const float p2 = ex2_approx(fmaf(__uint_as_float(s2[c + 2]), c_row, bias));
        const float p3 = ex2_approx(fmaf(__uint_as_float(s2[c + 3]), c_row, bias));
        sum += (p0 + p1) + (p2 + p3);
        pk[8 + c / 4] = pack_e4m3x4(p0, p1, p2, p3);
      }
      // P and O are free once the block before's P.V completed
      if (h >= 1 && !warp_spin(&bars->pv_done, (h - 1) & 1, abort_flag, __LINE__)) {
        ok = false;
        break;
      }
      {  // this thread's 64 keys of row r: 16-byte chunks 4 hf .. 4 hf + 3
        uint8_t* lp = smem + kOffP + prow;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(lp + (4 * hf + q) * kPLbo) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
      fence_proxy_async_smem();
      rescale_to(m_new, first);
      l_run += sum;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);  // P written and O rescaled
      if (!pc.last()) continue;

      // ---- segment end ----
      const int sp = cur_seg & 1;
      bars->xsum[sp][hf][r] = l_run;
      if (!xsync()) {
        ok = false;
        break;
      }
      const float l_tot = (bars->xsum[sp][0][r] + bars->xsum[sp][1][r]) * (1.0f / kPScale);  // sum of p
      const bool whole = (pc.sg.lo == 0 && pc.sg.hi == pc.sg.n);
      const float o_scale = kv_scale / kPScale;  // tensor-core units -> true units
      const float f = whole ? ((l_tot > 0.f) ? o_scale / l_tot : 0.f) : o_scale;
      const int slot = whole ? 0 : prm.num_splits[pc.sg.b] + pc.sg.split;
      // O is final once the P.V of the segment's last block completed
      if (!warp_wait(&bars->pv_done, h & 1, abort_flag, __LINE__)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int col0 = part * 256 + hf * kOHalf;       // this thread's O columns
      const int grow = (warp % 4) * 32 + (lane & ~3);  // the lane group's first row
      uint16_t* obase = whole ? prm.out + static_cast<size_t>(pc.sg.b) * R * kDV
                              : prm.ws_o + static_cast<size_t>(slot) * kRows * kDV;
#pragma unroll 1
      for (int ch = 0; ch < kOHalf / 32; ++ch) {
        uint32_t o[32];
        tmem_ld32(lane_base + kTO + hf * kOHalf + ch * 32, o);
        tmem_ld_wait();
        uint4 pcs[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          pcs[c].x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * f, __uint_as_float(o[8 * c + 1]) * f);
          pcs[c].y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * f, __uint_as_float(o[8 * c + 3]) * f);
          pcs[c].z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * f, __uint_as_float(o[8 * c + 5]) * f);
          pcs[c].w = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * f, __uint_as_float(o[8 * c + 7]) * f);
        }
        lane_group_transpose<4>(pcs, lane);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          if (grow + kk < R)
            *reinterpret_cast<uint4*>(obase + static_cast<size_t>(grow + kk) * kDV + col0 + ch * 32 +
                                      8 * (lane & 3)) = pcs[kk];
      }
      tc_fence_before();  // O is overwritten by the next segment's first P.V after the next p_full
      if (r < R && part == 0 && hf == 0) {  // the row's (uncorrected) LSE, or the piece's (m, l)
        if (whole) {
          prm.lse[static_cast<size_t>(pc.sg.b) * R + r] = (l_tot > 0.f) ? (m_run + lg2_approx(l_tot)) * kLn2 : kNegInf;
        } else {
          prm.ws_ml[static_cast<size_t>(slot) * kRows + r] = make_float2((l_tot > 0.f) ? m_run : kNegInf, l_tot);
        }
      }
    }
    if (!ok && lane == 0) *abort_flag = 1u;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_fp8(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const MlaParams& prm, int num_units,
                       cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};  // per device: CUDA keeps the limit per device
  const cudaError_t e = configure_once(configured, [] {
    return cudaFuncSetAttribute(mla_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(f8::smem_bytes()));
  });
  if (e != cudaSuccess) return e;
  return launch_dependent(mla_fp8_kernel, dim3(num_units * 2), dim3(f8::kThreads), f8::smem_bytes(), stream, tm_lat,
                          tm_rope, prm);
}

cudaError_t launch_16bit(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const MlaParams& prm, int num_units,
                         cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};  // per device: CUDA keeps the limit per device
  const cudaError_t e = configure_once(configured, [] {
    return cudaFuncSetAttribute(mla_decode_16bit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem_bytes16()));
  });
  if (e != cudaSuccess) return e;
  return launch_dependent(mla_decode_16bit_kernel, dim3(num_units * Cfg16::kParts), dim3(Cfg16::kThreads),
                          smem_bytes16(), stream, tm_lat, tm_rope, prm);
}

}  // namespace mla

cudaError_t launch_mla_decode_fp8(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const MlaParams& prm,
                                  int num_units, cudaStream_t stream) {
  return mla::launch_fp8(tm_lat, tm_rope, prm, num_units, stream);
}

cudaError_t launch_mla_decode_16bit(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const MlaParams& prm,
                                    int num_units, cudaStream_t stream) {
  return mla::launch_16bit(tm_lat, tm_rope, prm, num_units, stream);
}

cudaError_t launch_mla_qprep(const MlaParams& prm, cudaStream_t stream) {
  if (prm.b == 0) return cudaSuccess;
  return launch_dependent(mla::f8::mla_qprep_kernel, dim3(prm.b, mla::kRows / 32), dim3(256), 0, stream, prm);
}

cudaError_t mla_set_wait_test(int fault_page, uint64_t wait_limit_ns) {
  const uint64_t limit = wait_limit_ns ? wait_limit_ns : kWaitLimitNs;
  cudaError_t e = cudaMemcpyToSymbol(mla::f8::g_fault_page, &fault_page, sizeof(fault_page));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_wait_limit_ns, &limit, sizeof(limit));
  return e;
}

void mla_read_and_clear_timeout_site(uint32_t where[3]) {
  uint32_t v[4] = {0, 0, 0, 0}, z[4] = {0, 0, 0, 0};
  cudaMemcpyFromSymbol(v, g_timeout_where, sizeof(v));
  cudaMemcpyToSymbol(g_timeout_where, z, sizeof(z));
  for (int i = 0; i < 3; ++i) where[i] = v[3] ? v[i] : 0u;
}

uint32_t mla_read_and_clear_status() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_mla, sizeof(v));
  cudaMemcpyToSymbol(g_status_mla, &z, sizeof(z));
  return v;
}

}  // namespace fp8mla
