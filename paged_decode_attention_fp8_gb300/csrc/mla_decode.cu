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

// kCluster: the barrier also receives arrivals from the other CTA of a cluster
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
            waited = use == 0 || wait_bounded(&bars->kv_empty[st], (use - 1) & 1, abort_flag, &g_status_mla);
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
        wait_bounded(&bars->kv_full[j % C::kStages], (j / C::kStages) & 1, nullptr, &g_status_mla);
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
        if (!wait_bounded(&bars->p_full, j & 1, abort_flag, &g_status_mla)) return false;
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
        if (!wait_bounded(&bars->q_full, seg_i & 1, abort_flag, &g_status_mla)) break;
        const int first_i = i;
        for (int pg = sg.lo; pg < sg.hi; ++pg, ++i) {
          const int st = i % C::kStages;
          const int use = i / C::kStages;
          if (!wait_bounded(&bars->kv_full[st], use & 1, abort_flag, &g_status_mla) ||
              !wait_bounded(&bars->cvt_ready[st], use & 1, abort_flag, &g_status_mla) ||
              (i > 0 && !wait_bounded(&bars->s_free, (i - 1) & 1, abort_flag, &g_status_mla))) {
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
      wait_bounded(&bars->final_mma, 0, nullptr, &g_status_mla);
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
        if (t == 0) bars->cvt_ok = wait_bounded(&bars->kv_full[st], use & 1, abort_flag, &g_status_mla) ? 1u : 0u;
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
      const bool ok = warp_wait(&bars->xchg, xphase & 1, abort_flag);
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
        if (!warp_wait(&bars->s_full, i & 1, abort_flag)) {
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

        if (i > 0 && !warp_wait(&bars->pv_done, (i - 1) & 1, abort_flag)) {
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
      if (!warp_wait(&bars->pv_done, (i - 1) & 1, abort_flag)) break;
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
// Q preparation for FP8 dots (one grid ahead of the decode kernel).
// ===========================================================================
namespace f8 {
// Quantised Q of a sequence (FP8 dots), as written by mla_qprep_kernel: two
// latent slots, slot h (h = 0, 1) holding per row latent bytes [256 h,
// 256 h + 256) at a 272-byte pitch, then the RoPE values as f16 at a 144-byte
// pitch (pitches chosen so a quarter-warp's 16-byte row accesses hit distinct
// banks), then the latent quantisation error q_hat qs - q, 128 rows x 512
// bf16, read by the combine kernel for the LSE correction.
constexpr int kQLatPitch = 272;
constexpr int kQRopePitch = 144;
constexpr int kQLatSlotBytes = kRows * kQLatPitch;
constexpr int kQRopeSlotBytes = kRows * kQRopePitch;
constexpr int kQErrOff = 2 * kQLatSlotBytes + kQRopeSlotBytes;
static_assert(kQErrOff == kMlaQErrOff && kQErrOff + kRows * kDLat * 2 == kMlaQBytes, "quantised-Q layout");
static_assert(kQLatPitch % 16 == 0 && kQRopePitch % 16 == 0 && kQLatSlotBytes % 16 == 0, "16-byte rows");

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

// ===========================================================================
// FP8-dots kernel: one work unit = a cluster of two CTAs.
//
// CTA `rank` (0 or 1) owns dv columns [256 rank, 256 rank + 256) of O, and
// the unit's pages alternate between the two CTAs: page g of the unit's page
// stream (counted across its segments) belongs to CTA g % 2.  The owner of a
// page computes its scores S = Q K^T and its probabilities P; the other CTA
// only multiplies P by its own dv half of the page's V.  P (128 rows x 64
// keys, E4M3) and the running row maximum that P was computed against travel
// to the other CTA through distributed shared memory, so each page's Q.K^T
// and softmax run once per unit (the pair no longer repeats them).
//
// Page g's P is taken against a reference m_g (log2 units) that the owner
// decides from what it already has: m_g = max(m_{g-2}, m_{g-3}) (its own
// previous page's reference and the other CTA's reference of page g - 3,
// within the segment), raised to page g's row maximum when that exceeds it by
// more than kTau.  m_g travels with P; both CTAs rescale their O halves and
// row sums to m_g before page g's P.V, so both apply the same factors in the
// same order (a factor may be above 1 for a page after the other CTA raised
// its reference), every stored P is at most 64 * 2^kTau < 448, and no page
// waits for the other CTA's decision on the page just before it.
//
// Per CTA: TMEM holds its O half (256 columns), two S buffers (64 each; its
// own pages alternate, so one page's Q.K^T runs while the softmax works on
// the previous one) and the latent Q (128, E4M3).  Shared memory holds a V
// ring with this CTA's dv half of the latent bytes of every page (6 x 16 KB,
// released by the page's P.V), a K ring with the rest of this CTA's own pages
// (3 x 24 KB: the other latent half and the RoPE part, converted to f16 in
// place; released when the page's Q.K^T completes -- Q.K^T reads the page's
// latent bytes from both rings), Q's RoPE part (f16, 16 KB) and four P
// messages: page g's P and its 128 row references go to message g % 4 in
// both CTAs (to the other CTA by asynchronous remote stores that count their
// bytes on its p_rx barrier; the sender does not wait for them), and a
// message is rewritten four pages later, after both CTAs' P.V of the page
// before read it.
// ===========================================================================
namespace pr {
constexpr int kKStages = 3;   // own pages: the other latent half and the RoPE part, for Q.K^T
constexpr int kVStages = 6;   // this CTA's latent half of every page, for P.V (and own pages' Q.K^T)
constexpr int kThreads = 384;
// a K stage: the other CTA's two 128-byte latent boxes, then the RoPE part as
// f16 (64 keys x 128 B, 128-byte swizzle), converted in place from the E4M3
// RoPE box that the load puts in the second half of that region
constexpr int kKRope = 2 * kLatBox;
constexpr int kKRopeRaw = kKRope + kPage * 64;
constexpr int kKBytes = kKRope + kLatBox;
constexpr uint32_t kKTx = 2 * kLatBox + kPage * 64;   // bytes the K part of an own page's load delivers
constexpr int kVBytes = 2 * kLatBox;                  // latent bytes [256 rank, 256 rank + 256) of a page
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKStages * kKBytes;
constexpr int kOffQRope = kOffV + kVStages * kVBytes;  // Q RoPE, 128 rows x 64 f16, 128-byte swizzle
constexpr int kOffP = kOffQRope + kRows * 128;         // four P messages
constexpr int kPBytes = kRows * kPage;                 // P: 128 rows x 64 E4M3 keys
constexpr int kPTile = kPBytes + kRows * 4;            // then the 128 row references (float)
constexpr int kPTiles = 4;
static_assert(kPTile % 128 == 0, "16-byte aligned P tiles and reference pieces");
constexpr int kSmemData = kOffP + kPTiles * kPTile;
// P: 8-row x 16-byte core matrices, key chunk c of row group G at c * kPLbo + G * kPSbo, so the 32
// rows x 16 bytes that one warp writes per key chunk are one contiguous 512-byte piece
constexpr int kPLbo = 2048, kPSbo = 128;
constexpr float kPScale = 64.0f, kPLog2 = 6.0f;  // P is stored as E4M3(64 p)
constexpr float kTau = 2.75f;                    // 64 * 2^2.75 = 430.5 < 448
// TMEM columns: O half, two S buffers, Q latent (E4M3, the A operand of the latent Q.K^T)
constexpr uint32_t kTO = 0, kTS = 256, kTQ = 384;
static_assert(kKBytes % 1024 == 0 && kOffV % 1024 == 0 && kVBytes % 1024 == 0 && kOffP % 1024 == 0 &&
                  kKRope % 1024 == 0 && kOffQRope % 1024 == 0,
              "1 KB aligned tiles");

struct Bars {
  uint64_t k_full[kKStages];        // own page's other latent half and RoPE part loaded
  uint64_t k_cvt[kKStages];         // its RoPE part converted to f16
  uint64_t k_empty[kKStages];       // its Q.K^T completed: the stage may be refilled
  uint64_t v_full[kVStages];        // by page g % kVStages: this CTA's latent half of page g loaded
  uint64_t v_empty[kVStages];       // its P.V (and for an own page its Q.K^T) completed
  uint64_t s_full[2];               // by own-page parity: S buffer holds the page's scores
  uint64_t s_free[2];               // S buffer read out (8 softmax warps)
  uint64_t p_full[kPTiles];         // by tile: P written here (own page) / O ready here (other's page)
  uint64_t p_rx[2];                 // by tile (g / 2 % 2): the other CTA's P message copied in
                                    // (transaction bytes; re-armed by a softmax thread)
  uint64_t pv_done[kPTiles];        // by tile: the P.V of the page completed here -- and, for the tiles of
                                    // this CTA's pages (g % 2 = rank), in the other CTA too (2 arrivals)
  uint64_t lx_full[2];              // by segment parity: the other CTA's row sums arrived (4 warps)
  uint64_t q_full;                  // a segment's Q copied in (8 softmax warps)
  uint64_t final_mma, xchg;
  uint32_t tmem_base, abort_flag, cvt_ok;
  // written by 16-byte stores (the other CTA's lane 0 sends 32 rows at a time)
  alignas(16) float lx[2][kRows];   // the other CTA's row sums, by segment parity
  float xsum[2][2][kRows];          // by segment parity: row-sum halves of the two softmax threads of a row
};
static_assert(offsetof(Bars, lx) % 16 == 0, "16-byte rows of sums");
static_assert(kSmemData % 16 == 0, "the barrier block starts 16-byte aligned");

constexpr size_t smem_bytes() { return kSmemData + sizeof(Bars) + 1024; }
static_assert(smem_bytes() <= 232448, "fits the 227 KB opt-in shared memory of a CTA");

// Pages of a unit one at a time: g counts the unit's pages across segments,
// seg its non-empty segments.
struct PageCursor {
  SegmentWalker walk;
  Segment sg;
  int pg = 0, g = -1, seg = -1;
  bool valid = false;
  __device__ PageCursor(const MlaParams& p, int unit) : walk(p, unit) {}
  __device__ bool next() {
    if (valid && pg + 1 < sg.hi) {
      ++pg;
      ++g;
      return true;
    }
    valid = walk.next(sg);
    if (!valid) return false;
    pg = sg.lo;
    ++g;
    ++seg;
    return true;
  }
  __device__ bool first() const { return pg == sg.lo; }
  __device__ bool last() const { return pg == sg.hi - 1; }
};

// Unit-level fault injection for the bounded-wait test: when g_fault_page is
// p + 1, CTA 0 of unit 0 never issues the loads of its page p, so every wait
// on them runs out (see fp8mla_test_fault_injection).
__device__ int g_fault_page = 0;

}  // namespace pr

__global__ void __launch_bounds__(pr::kThreads, 1)
    mla_fp8_pair_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope,
                        const MlaParams prm) {
  using namespace pr;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + kSmemData);
  volatile uint32_t* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int unit = blockIdx.x / 2;
  const uint32_t rank = cluster_ctarank();
  const uint32_t other = rank ^ 1u;
  auto remote = [&](const void* p) { return mapa_shared(smem_u32(p), other); };
  // stop this CTA and tell the other one, whose waits then end too
  auto fail = [&]() {
    *abort_flag = 1u;
    st_cluster_u32(remote(&bars->abort_flag), 1u);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_cvt[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], kSoftmaxThreads / 32);
    }
    for (int b = 0; b < kPTiles; ++b) {
      mbar_init(&bars->p_full[b], kSoftmaxThreads / 32);
      mbar_init(&bars->pv_done[b], (b & 1) == static_cast<int>(rank) ? 2 : 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&bars->p_rx[b], 1);
    for (int b = 0; b < 2; ++b) mbar_init(&bars->lx_full[b], kSoftmaxThreads / 64);
    mbar_init(&bars->q_full, kSoftmaxThreads / 32);
    mbar_init(&bars->final_mma, 1);
    mbar_init(&bars->xchg, kSoftmaxThreads / 32);
    bars->abort_flag = 0;
    fence_barrier_init();
    for (int b = 0; b < 2; ++b) mbar_arrive_expect_tx(&bars->p_rx[b], kPTile);  // the first two messages
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
  // both CTAs' barriers are initialised before either arrives on the other's
  cluster_arrive();
  cluster_wait();
  griddep_launch_dependents();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer ----
    // Two streams of loads, issued by lane 0 as their stages free up (own pages
    // first).  Own page g: its latent half [256 rank, +256) into V stage
    // g % kVStages, the other half and the RoPE box into the next K stage.  The
    // other CTA's page g: this CTA's latent half into V stage g % kVStages.
    // Each stream fetches the block-table entry of its next page right after
    // issuing a load, so the entry is at hand when the stages free up.
    if (lane == 0) {
      tma_prefetch_desc(&tm_lat);
      tma_prefetch_desc(&tm_rope);
      const int fault = (unit == 0 && rank == 0) ? *(volatile int*)&g_fault_page : 0;
      auto phys_of = [&](const PageCursor& c) -> int {
        int ph = __ldg(prm.block_table + static_cast<size_t>(c.sg.b) * prm.max_pages + c.pg);
        if (ph < 0 || ph >= prm.num_pages) {
          atomicOr(&g_status_mla, FP8MLA_DEV_BAD_PAGE);
          ph = 0;
        }
        return ph;
      };
      PageCursor oc(prm, unit), xc(prm, unit);  // own pages; the other CTA's pages
      auto advance = [&](PageCursor& c, int want) -> bool {
        while (c.next())
          if ((c.g & 1) == want) return true;
        return false;
      };
      bool o_more = advance(oc, static_cast<int>(rank)), x_more = advance(xc, static_cast<int>(other));
      int o_phys = o_more ? phys_of(oc) : 0, x_phys = x_more ? phys_of(xc) : 0;
      int kn = 0;  // own-page loads issued
      uint32_t v_last = 0, v_par = 0, k_last = 0, k_par = 0;  // per stage: loaded here, and its phase parity
      auto v_free = [&](int g) { return g < kVStages || mbar_test_wait(&bars->v_empty[g % kVStages], ((g / kVStages) - 1) & 1); };
      auto load_v = [&](int g, int phys) {
        const int st = g % kVStages;
        uint8_t* sb = smem + kOffV + st * kVBytes;
        mbar_arrive_expect_tx(&bars->v_full[st], kVBytes);
        tma_load_3d(sb, &tm_lat, &bars->v_full[st], static_cast<int>(rank) * 256, 0, phys);
        tma_load_3d(sb + kLatBox, &tm_lat, &bars->v_full[st], static_cast<int>(rank) * 256 + 128, 0, phys);
        v_last |= 1u << st;
        v_par = (v_par & ~(1u << st)) | (static_cast<uint32_t>((g / kVStages) & 1) << st);
      };
      uint32_t polls = 0;
      uint64_t t_idle = 0;
      bool ok = true;
      while (ok && (o_more || x_more)) {
        bool did = false;
        if (o_more) {
          const int st = kn % kKStages, use = kn / kKStages;
          if ((use == 0 || mbar_test_wait(&bars->k_empty[st], (use - 1) & 1)) && v_free(oc.g)) {
            if (fault != oc.g + 1) {
              load_v(oc.g, o_phys);
              uint8_t* sb = smem + kOffK + st * kKBytes;
              mbar_arrive_expect_tx(&bars->k_full[st], kKTx);
              tma_load_3d(sb, &tm_lat, &bars->k_full[st], static_cast<int>(other) * 256, 0, o_phys);
              tma_load_3d(sb + kLatBox, &tm_lat, &bars->k_full[st], static_cast<int>(other) * 256 + 128, 0, o_phys);
              tma_load_3d(sb + kKRopeRaw, &tm_rope, &bars->k_full[st], kDLat, 0, o_phys);
              k_last |= 1u << st;
              k_par = (k_par & ~(1u << st)) | (static_cast<uint32_t>(use & 1) << st);
            }
            ++kn;
            o_more = advance(oc, static_cast<int>(rank));
            if (o_more) o_phys = phys_of(oc);
            did = true;
          }
        }
        if (!did && x_more && v_free(xc.g)) {
          if (fault != xc.g + 1) load_v(xc.g, x_phys);
          x_more = advance(xc, static_cast<int>(other));
          if (x_more) x_phys = phys_of(xc);
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
      if (!ok) fail();
      // Never leave with copies in flight: wait for the last load of each stage.
      for (int st = 0; st < kKStages; ++st)
        if ((k_last >> st) & 1u) wait_bounded(&bars->k_full[st], (k_par >> st) & 1u, nullptr, &g_status_mla, __LINE__);
      for (int st = 0; st < kVStages; ++st)
        if ((v_last >> st) & 1u) wait_bounded(&bars->v_full[st], (v_par >> st) & 1u, nullptr, &g_status_mla, __LINE__);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer ----
    // The whole warp runs the loop and one elected lane issues.  The warp
    // polls the conditions of the next own page's Q.K^T and of the next
    // page's P.V and issues whichever is ready (the Q.K^T first), so neither
    // waits behind the other.  Q.K^T(j) needs S buffer j % 2 read out (own
    // page j - 2's scores), its page loaded and converted and, when it opens a
    // segment, that segment's Q; P.V(g) needs P(g) written and O ready, and
    // the page's V half loaded.  Before the P.V of a sequence's last page the
    // warp zeroes the V rows past the sequence end (they may hold anything,
    // and P is 0 there).
    constexpr uint32_t idesc8 = make_idesc(0, 0, 0, 0, 64, 128);    // e4m3 x e4m3, both K-major, N = 64
    constexpr uint32_t idesc16 = make_idesc(0, 0, 0, 0, 64, 128);   // f16 x f16 (E4M3 keys are exact in f16)
    constexpr uint32_t idesc_pv = make_idesc(0, 0, 0, 1, 256, 128); // e4m3, B MN-major, N = 256
    const bool leader = elect_one();
    const uint16_t other_mask = static_cast<uint16_t>(1u << other);
    const uint64_t qd = make_sdesc(smem_u32(smem + kOffQRope), 16, 1024, SWIZZLE_128B);
    PageCursor qk(prm, unit);  // next own page whose Q.K^T is due
    PageCursor pv(prm, unit);  // next page whose P.V is due
    int qn = 0, qk_seg = -1, qk_n = 0;  // Q copies consumed, segment of the last Q.K^T, Q.K^Ts issued
    auto qk_advance = [&]() -> bool {
      while (qk.next())
        if ((qk.g & 1) == static_cast<int>(rank)) return true;
      return false;
    };
    bool qk_more = qk_advance();
    bool pv_more = pv.next();
    bool ok = true;
    uint64_t t_idle = 0;
    uint32_t polls = 0;
    while (ok && (qk_more || pv_more)) {
      bool did = false;
      if (qk_more) {
        const int j = qk_n;  // own pages in order
        const int st = j % kKStages;
        const bool opens = qk.seg != qk_seg;
        // (its V-stage probe comes after the K-stage one: a converted K part means the
        // page's load was issued, so the V stage's previous phase has completed)
        const int vst = qk.g % kVStages;
        const bool ready = (!opens || mbar_test_wait(&bars->q_full, qn & 1)) &&
                           (j < 2 || mbar_test_wait(&bars->s_free[j & 1], ((j - 2) >> 1) & 1)) &&
                           mbar_test_wait(&bars->k_cvt[st], (j / kKStages) & 1) &&
                           mbar_test_wait(&bars->v_full[vst], (qk.g / kVStages) & 1);
        if (__all_sync(0xffffffffu, ready)) {
          if (opens) {
            qk_seg = qk.seg;
            ++qn;
          }
          ++qk_n;
          tc_fence_after();
          const uint32_t t_s = tmem + kTS + (j & 1) * kPage;
          const uint32_t kb = smem_u32(smem + kOffK + st * kKBytes);
          // latent box q (128 bytes of each key row) is in the V stage for this CTA's half, else in the K stage
          const uint64_t kd = make_sdesc(kb, 16, 1024, SWIZZLE_128B);
          const uint64_t vd = make_sdesc(smem_u32(smem + kOffV + vst * kVBytes), 16, 1024, SWIZZLE_128B);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const int q = kk >> 2;
            const uint64_t bd = ((q >> 1) == static_cast<int>(rank)) ? vd + (((q & 1) * kLatBox + (kk & 3) * 32) >> 4)
                                                                     : kd + (((q & 1) * kLatBox + (kk & 3) * 32) >> 4);
            mma_f8_ts_if(leader, t_s, tmem + kTQ + kk * 8, bd, idesc8, kk > 0 ? 1u : 0u);
          }
          const uint64_t rd = make_sdesc(kb + kKRope, 16, 1024, SWIZZLE_128B);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_f16_ss_if(leader, t_s, qd + ((kk * 32) >> 4), rd + ((kk * 32) >> 4), idesc16, 1u);
          tc_commit_if(leader, &bars->s_full[j & 1]);
          tc_commit_if(leader, &bars->k_empty[st]);
          qk_more = qk_advance();
          did = true;
        }
      }
      if (!did && pv_more) {
        const int g = pv.g;
        const bool mine = (g & 1) == static_cast<int>(rank);
        const int idx = g >> 1;
        const int st = g % kVStages;
        // P(g) written here (own page) or O ready for it here (the other CTA's
        // page; its P message arrived before that), and the V half loaded
        const bool ready = mbar_test_wait(&bars->p_full[g & 3], (g >> 2) & 1) &&
                           mbar_test_wait(&bars->v_full[st], (g / kVStages) & 1);
        if (__all_sync(0xffffffffu, ready)) {
          uint8_t* vs = smem + kOffV + st * kVBytes;
          const int live = pv.sg.s_k - pv.pg * kPage;  // rows of the page that hold keys
          if (pv.pg == pv.sg.n - 1 && live < kPage) {  // zero the rows past the sequence end
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int i = lane; i < (kPage - live) * 16; i += 32) {
              const int row = live + i / 16, c = i % 16;
              *reinterpret_cast<uint4*>(vs + (c >> 3) * kLatBox + row * 128 + ((c & 7) << 4)) = z;
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          tc_fence_after();
          const uint64_t pd = make_sdesc(smem_u32(smem + kOffP + (g & 3) * kPTile), kPLbo, kPSbo, SWIZZLE_NONE);
          const uint64_t vd = make_sdesc(smem_u32(vs), kLatBox, 1024, SWIZZLE_128B);
          const bool first = pv.first();
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma_f8_ss_if(leader, tmem + kTO, pd + ((kk * 2 * kPLbo) >> 4), vd + ((kk * 4096) >> 4), idesc_pv,
                         (first && kk == 0) ? 0u : 1u);
          tc_commit_if(leader, &bars->pv_done[g & 3]);
          tc_commit_if(leader, &bars->v_empty[st]);
          // the other CTA's page: its owner may reuse the tile once both P.Vs completed
          if (!mine) tc_commit_mc_if(leader, &bars->pv_done[g & 3], other_mask);
          pv_more = pv.next();
          did = true;
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
    if (!ok) fail();
    if (leader) tc_commit(&bars->final_mma);
    __syncwarp();
    warp_wait(&bars->final_mma, 0, nullptr, __LINE__);
  } else if (warp == 2 || warp == 3) {
    // ---------------------- RoPE conversion of own pages (64 threads) ----
    // Thread t reads the E4M3 RoPE bytes of token row t from the second half
    // of the stage's RoPE region, and after all have read, writes them as f16
    // (exact) over the whole region, 128-byte swizzled; rows past the sequence
    // end become 0 (their scores are masked anyway).
    const int t = threadIdx.x - 64;  // token row of the page
    PageCursor pc(prm, unit);
    bool ok = true;
    int j = 0;
    while (ok && pc.next()) {
      if ((pc.g & 1) != static_cast<int>(rank)) continue;
      const int st = j % kKStages, use = j / kKStages;
      ++j;
      if (t == 0)
        bars->cvt_ok = wait_bounded(&bars->k_full[st], use & 1, abort_flag, &g_status_mla, __LINE__) ? 1u : 0u;
      named_bar_sync(1, 64);
      if (!bars->cvt_ok) {
        ok = false;
        break;
      }
      uint8_t* kb = smem + kOffK + st * kKBytes;
      const bool dead = (pc.pg == pc.sg.n - 1) && (t >= pc.sg.s_k - pc.pg * kPage);  // slot past the end
      const uint4 z = make_uint4(0, 0, 0, 0);
      uint4 raw[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) raw[c] = dead ? z : reinterpret_cast<const uint4*>(kb + kKRopeRaw + t * 64)[c];
      named_bar_sync(1, 64);  // every raw row is read before the f16 rows overwrite them
      const int sw = t & 7;
      uint8_t* dst = kb + kKRope + t * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 v = raw[c];
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
      fence_proxy_async_smem();
      named_bar_sync(1, 64);
      if (t == 0) mbar_arrive(&bars->k_cvt[st]);
    }
    if (!ok && t == 0) fail();
  } else {
    // ------------------ softmax / Q copy / epilogue (8 warps, 2 per row) ----
    const int hf = (warp - 4) / 4;         // which half of the row
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
    const uint32_t r_lx = remote(&bars->lx[0][r]);
    const uint32_t r_prx0 = remote(&bars->p_rx[0]);
    const uint32_t r_lxfull0 = remote(&bars->lx_full[0]);
    const uint32_t r_p0 = remote(smem + kOffP);
    const uint32_t prow = static_cast<uint32_t>((r >> 3) * kPSbo + (r & 7) * 16);
    // Sends the 32 values v of this warp's rows (rows 32 (warp % 4) .. + 31) to
    // the other CTA at cluster address dst and arrives on its barrier rbar:
    // lane 0 gathers them and stores them itself, so that its release covers
    // every value (other lanes' remote stores would not be ordered by it).
    auto send_rows = [&](uint32_t dst, float v, uint32_t rbar) {
      uint4 w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        w[i].x = __float_as_uint(__shfl_sync(0xffffffffu, v, 4 * i));
        w[i].y = __float_as_uint(__shfl_sync(0xffffffffu, v, 4 * i + 1));
        w[i].z = __float_as_uint(__shfl_sync(0xffffffffu, v, 4 * i + 2));
        w[i].w = __float_as_uint(__shfl_sync(0xffffffffu, v, 4 * i + 3));
      }
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) st_cluster_v4(dst + 16 * i, w[i]);
        mbar_arrive_cluster(rbar, 1);
      }
    };

    // Copies this half of sequence b_seq's quantised Q row (prepared by
    // mla_qprep_kernel) in: latent bytes [256 hf, +256) into TMEM columns
    // kTQ + 64 hf.., RoPE values [32 hf, +32) into the Q RoPE tile.
    int qn = 0;
    float qs_cur = 1.f;
    auto copy_q = [&](int b_seq) -> bool {
      const uint8_t* qb = prm.qbuf + static_cast<size_t>(b_seq) * kMlaQBytes;
      const uint4* lat = reinterpret_cast<const uint4*>(qb + hf * f8::kQLatSlotBytes + r * f8::kQLatPitch);
      const uint4* rope = reinterpret_cast<const uint4*>(qb + 2 * f8::kQLatSlotBytes + r * f8::kQRopePitch + hf * 64);
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
      ++qn;
      return true;
    };
    // true if some segment after the cursor's holds a page of this CTA; its sequence in *b_out
    auto next_q_segment = [&](const PageCursor& at, int* b_out) -> bool {
      SegmentWalker peek = at.walk;
      Segment nx;
      int g0 = at.g + (at.sg.hi - at.pg);  // unit index of the next segment's first page
      while (peek.next(nx)) {
        const int n = nx.hi - nx.lo;
        if (n >= 2 || (g0 & 1) == static_cast<int>(rank)) {
          *b_out = nx.b;
          return true;
        }
        g0 += n;
      }
      return false;
    };

    PageCursor pc(prm, unit);
    bool ok = true;
    int cur_seg = -1;
    float m_run = kNegInf, l_run = 0.f;  // reference of O and l; this CTA's share of l
    float m_own = kNegInf;                // this CTA's latest reference in the segment
    int pend = -1;  // the other CTA's page whose rescale / O-ready is still due
    bool pend_first = false;
    int qtok = 0, visible = 0, min_visible = 0;
    float c_row = 0.f;

    // Moves O and l to a new reference before a page's P.V: both are
    // multiplied by 2^(m_run - m_new) once the P.V of page g - 1 completed.
    // A reference of -inf (the row sees no key of the page, so its P is 0)
    // leaves them where they are, in both CTAs alike.
    auto rescale_to = [&](int g, float m_new, bool first) -> bool {
      const bool rescale = !first && m_new != m_run && m_new != kNegInf;
      const float alpha = rescale ? ex2_approx(m_run - m_new) : 1.f;
      l_run = first ? 0.f : l_run * alpha;
      if (first || rescale) m_run = m_new;
      if (__any_sync(0xffffffffu, rescale)) {
        if (!warp_spin(&bars->pv_done[(g - 1) & 3], ((g - 1) >> 2) & 1, abort_flag, __LINE__)) return false;
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
      return true;
    };
    // The other CTA's page g: wait for its P message, take the reference it
    // carries (kept for this CTA's page g + 3), rescale O and l to it, and
    // declare O ready for the page's P.V.
    float m_other = kNegInf;  // the other CTA's latest reference in this segment
    auto finish_other = [&](int g, bool first) -> bool {
      const int k = g >> 1;
      if (!warp_spin(&bars->p_rx[k & 1], (k >> 1) & 1, abort_flag, __LINE__)) return false;
      fence_proxy_async_smem();  // the remotely stored P is read by this CTA's P.V
      // (every softmax thread has passed this phase before the message's next
      // bytes can come: they follow this page's P.V here)
      if (warp == 4 && lane == 0) mbar_arrive_expect_tx(&bars->p_rx[k & 1], kPTile);
      const float m_new = reinterpret_cast<const float*>(smem + kOffP + (g & 3) * kPTile + kPBytes)[r];
      m_other = m_new;
      // (this CTA's arrival for page g comes after page g - 4's phase of the tile
      // completed: the message's sender waited for this CTA's P.V of page g - 4)
      if (!rescale_to(g, m_new, first)) return false;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[g & 3]);
      return true;
    };

    // Q of the first segment holding a page of this CTA
    {
      PageCursor probe(prm, unit);
      if (probe.next()) {
        int bq = probe.sg.b;
        const int n = probe.sg.hi - probe.sg.lo;
        bool have = n >= 2 || (probe.g & 1) == static_cast<int>(rank);
        if (!have) have = next_q_segment(probe, &bq);
        if (have) {
          ok = copy_q(bq);
        }
      }
    }

    while (ok && pc.next()) {
      const int g = pc.g;
      if (pc.seg != cur_seg) {  // a new segment
        cur_seg = pc.seg;
        m_run = kNegInf;
        l_run = 0.f;
        m_own = kNegInf;
        m_other = kNegInf;
        qtok = (r < R) ? r / prm.h_q : 0;
        visible = prm.causal ? (pc.sg.s_k - prm.s_q + qtok + 1) : pc.sg.s_k;
        min_visible = prm.causal ? (pc.sg.s_k - prm.s_q + 1) : pc.sg.s_k;
        if (r < R && pc.first()) {  // warm L2 with the Q of the segment after this one
          int bn;
          if (next_q_segment(pc, &bn)) {
            const char* nq = reinterpret_cast<const char*>(prm.qbuf + static_cast<size_t>(bn) * kMlaQBytes);
            prefetch_l2(nq + hf * f8::kQLatSlotBytes + r * f8::kQLatPitch);
            prefetch_l2(nq + hf * f8::kQLatSlotBytes + r * f8::kQLatPitch + 128);
          }
        }
      }
      const bool mine = (g & 1) == static_cast<int>(rank);
      if (!mine) {
        pend = g;
        pend_first = pc.first();
      } else {
        const int j = g >> 1;
        c_row = prm.softmax_scale * kLog2e * qs_cur * kv_scale;
        if (!warp_spin(&bars->s_full[j & 1], (j >> 1) & 1, abort_flag, __LINE__)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // both halves of the row: the other half only for the row max
        uint32_t s[32], so[32];
        tmem_ld32(lane_base + kTS + (j & 1) * kPage + 32 * hf, s);
        tmem_ld32(lane_base + kTS + (j & 1) * kPage + 32 * (1 - hf), so);
        tmem_ld_wait();
        tc_fence_before();
        warp_arrive(&bars->s_free[j & 1]);  // own page j + 2's Q.K^T may overwrite this S buffer
        if (pc.pg * kPage + kPage > min_visible) {
          const int base = pc.pg * kPage + 32 * hf, base_o = pc.pg * kPage + 32 * (1 - hf);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (base + c >= visible) s[c] = __float_as_uint(kNegInf);
            if (base_o + c >= visible) so[c] = __float_as_uint(kNegInf);
          }
        }
        float m22[22];
#pragma unroll
        for (int c = 0; c < 10; ++c) {
          m22[c] = fmax3(__uint_as_float(s[3 * c]), __uint_as_float(s[3 * c + 1]), __uint_as_float(s[3 * c + 2]));
          m22[10 + c] =
              fmax3(__uint_as_float(so[3 * c]), __uint_as_float(so[3 * c + 1]), __uint_as_float(so[3 * c + 2]));
        }
        m22[20] = fmaxf(__uint_as_float(s[30]), __uint_as_float(s[31]));
        m22[21] = fmaxf(__uint_as_float(so[30]), __uint_as_float(so[31]));
        float m8[8];
#pragma unroll
        for (int c = 0; c < 7; ++c) m8[c] = fmax3(m22[3 * c], m22[3 * c + 1], m22[3 * c + 2]);
        m8[7] = m22[21];
        const float mx =
            fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * c_row;
        // P tile g % 4 is free once both CTAs' P.V of page g - 4 completed
        if (g >= 4 && !warp_spin(&bars->pv_done[g & 3], ((g - 4) >> 2) & 1, abort_flag, __LINE__)) {
          ok = false;
          break;
        }
        // the reference: this CTA's and the other's latest ones (pages g - 2 and g - 3),
        // raised to this page's maximum when that exceeds them by more than kTau
        const bool first = pc.first();
        const float m_known = fmaxf(m_own, m_other);
        const float m_new = (mx > m_known + kTau) ? mx : m_known;
        m_own = m_new;
        const float bias = (m_new == kNegInf) ? 0.f : (kPLog2 - m_new);
        float sum = 0.f;
        uint32_t pk[8];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(s[c]), c_row, bias));
          const float p1 = ex2_approx(fmaf(__uint_as_float(s[c + 1]), c_row, bias));
          const float p2 = ex2_approx(fmaf(__uint_as_float(s[c + 2]), c_row, bias));
          const float p3 = ex2_approx(fmaf(__uint_as_float(s[c + 3]), c_row, bias));
          sum += (p0 + p1) + (p2 + p3);
          pk[c / 4] = pack_e4m3x4(p0, p1, p2, p3);
        }
        {  // this thread's 32 keys of row r (16-byte chunks 2 hf, 2 hf + 1), and the row's reference,
           // here and (asynchronously, counted on its p_rx barrier) in the other CTA
          const uint32_t tile = static_cast<uint32_t>((g & 3) * kPTile);
          const uint4 a = make_uint4(pk[0], pk[1], pk[2], pk[3]), b2 = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          uint8_t* lp = smem + kOffP + tile + prow;
          *reinterpret_cast<uint4*>(lp + (2 * hf) * kPLbo) = a;
          *reinterpret_cast<uint4*>(lp + (2 * hf + 1) * kPLbo) = b2;
          const uint32_t rbar = r_prx0 + (j & 1) * 8;
          st_async_v4(r_p0 + tile + prow + (2 * hf) * kPLbo, a, rbar);
          st_async_v4(r_p0 + tile + prow + (2 * hf + 1) * kPLbo, b2, rbar);
          if (hf == 0) {
            reinterpret_cast<float*>(smem + kOffP + tile + kPBytes)[r] = m_new;
            st_async_f32(r_p0 + tile + kPBytes + r * 4, m_new, rbar);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        // the other CTA's previous page: O moves to its reference and is declared
        // ready for its P.V before this page's rescale
        if (pend >= 0) {
          if (!finish_other(pend, pend_first)) {
            ok = false;
            break;
          }
          pend = -1;
        }
        if (!rescale_to(g, m_new, first)) {
          ok = false;
          break;
        }
        l_run += sum;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[g & 3]);  // P written and O rescaled here
        // this CTA's last page of the segment: the next segment's Q may replace this one's
        bool last_own = pc.last() || (pc.pg + 1 == pc.sg.hi - 1);
        if (last_own) {
          int bn;
          if (next_q_segment(pc, &bn)) {
            ok = copy_q(bn);
          }
        }
      }
      if (!ok) break;
      if (!pc.last()) continue;

      // ---- segment end ----
      if (pend >= 0) {
        if (!finish_other(pend, pend_first)) {
          ok = false;
          break;
        }
        pend = -1;
      }
      // row sum: this CTA's two halves, then the other CTA's
      const int sp = cur_seg & 1;
      bars->xsum[sp][hf][r] = l_run;
      if (!xsync()) {
        ok = false;
        break;
      }
      const float l_here = bars->xsum[sp][0][r] + bars->xsum[sp][1][r];
      // one barrier per slot: the other CTA may finish the next segment before this one reads this slot
      if (hf == 0) send_rows(r_lx - lane * 4 + sp * kRows * 4, l_here, r_lxfull0 + sp * 8);
      if (!warp_wait<true>(&bars->lx_full[sp], (cur_seg >> 1) & 1, abort_flag, __LINE__)) {
        ok = false;
        break;
      }
      const float l_tot = (l_here + bars->lx[sp][r]) * (1.0f / kPScale);  // sum of p
      const bool whole = (pc.sg.lo == 0 && pc.sg.hi == pc.sg.n);
      const float o_scale = kv_scale / kPScale;  // tensor-core units -> true units
      const float f = whole ? ((l_tot > 0.f) ? o_scale / l_tot : 0.f) : o_scale;
      const int slot = whole ? 0 : prm.num_splits[pc.sg.b] + pc.sg.split;
      // O is final once this CTA's P.V of the segment's last page completed
      if (!warp_wait(&bars->pv_done[g & 3], (g >> 2) & 1, abort_flag, __LINE__)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int col0 = static_cast<int>(rank) * 256 + hf * kOHalf;  // this thread's O columns
      const int grow = (warp % 4) * 32 + (lane & ~3);                // the lane group's first row
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
        f8::lane_group_transpose<4>(pcs, lane);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          if (grow + kk < R)
            *reinterpret_cast<uint4*>(obase + static_cast<size_t>(grow + kk) * kDV + col0 + ch * 32 +
                                      8 * (lane & 3)) = pcs[kk];
      }
      tc_fence_before();  // O is overwritten by the next segment's first P.V after the next p_full
      if (r < R && rank == 0 && hf == 0) {  // the row's (uncorrected) LSE, or the piece's (m, l)
        if (whole) {
          prm.lse[static_cast<size_t>(pc.sg.b) * R + r] = (l_tot > 0.f) ? (m_run + lg2_approx(l_tot)) * kLn2 : kNegInf;
        } else {
          prm.ws_ml[static_cast<size_t>(slot) * kRows + r] = make_float2((l_tot > 0.f) ? m_run : kNegInf, l_tot);
        }
      }
    }
    if (!ok) fail();
    // The other CTA's P.V commits of this CTA's last pages arrive in this
    // CTA's shared memory: they must land before this CTA may exit.
    if (ok) {
      int last0 = -1, last1 = -1;  // last own page on each of this CTA's two tiles
      PageCursor cnt(prm, unit);
      while (cnt.next())
        if ((cnt.g & 1) == static_cast<int>(rank)) ((cnt.g >> 1) & 1 ? last1 : last0) = cnt.g;
      if (last0 >= 0) warp_spin(&bars->pv_done[last0 & 3], (last0 >> 2) & 1, abort_flag, __LINE__);
      if (last1 >= 0) warp_spin(&bars->pv_done[last1 & 3], (last1 >> 2) & 1, abort_flag, __LINE__);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // no CTA leaves while the other may still write to its shared memory
  cluster_arrive();
  cluster_wait();
}

cudaError_t launch_fp8(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const MlaParams& prm, int num_units,
                       cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};  // per device: CUDA keeps the limit per device
  const cudaError_t e = configure_once(configured, [] {
    return cudaFuncSetAttribute(mla_fp8_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(pr::smem_bytes()));
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_units * 2);
  cfg.blockDim = dim3(pr::kThreads);
  cfg.dynamicSmemBytes = pr::smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, mla_fp8_pair_kernel, tm_lat, tm_rope, prm);
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
