// Dense MLA decode over an E4M3 paged KV cache, tcgen05 + TMA, sm_103a.
//
// The operation (FlashMLA "update fp8 support", Improvements; test shape
// d = 576, dv = 512, h_kv = 1, s_q <= 2, causal) per sequence b:
//   S = Q K^T (Q: R = s_q * h_q rows x 576; K: the sequence's cached rows),
//   P = softmax(softmax_scale * S) under the causal mask, O = P V with V the
//   first 512 dims of the same rows; lse = log sum exp.
//
// GB300 design: one work unit = 2 CTAs of mla_fp8_kernel, each owning one
// 256-wide slice of dv.
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
//   * 16-bit dots run as two-term E4M3 dots: Q's latent part and P enter as
//     hi + lo (hi = E4M3(x), lo = E4M3(x - hi): bf16's 8 significant bits)
//     against the cache's exact E4M3 K and V, adding 16 Q_lo MMAs to each
//     Q.K^T and 2 P_lo MMAs to each P.V; the RoPE chunk is f16 as above.
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
//   * Rounding Q perturbs the LSE by softmax_scale * (q_hat - q) . k_mean,
//     where k_mean = sum_j p_j k_j; its latent part is exactly the output row,
//     so the combine kernel subtracts softmax_scale * (q_hat - q) . out, from
//     the finished output row and q_hat - q recomputed from q and the row's
//     scale with the decode kernel's rounding (one term or two).
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-3 page conversion (the RoPE part to f16) and tail zeroing,
// warps 4-11 softmax, Q copy and epilogue: query
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
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          uint32_t site = 0) {
  const bool ok = wait_bounded(bar, parity, abort_flag, &g_status_mla, site);
  return __all_sync(0xffffffffu, ok);
}

// warp_wait polling without suspension, for the waits on the per-page critical path
__device__ __forceinline__ bool warp_spin(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          uint32_t site = 0) {
  const bool ok = wait_spin(bar, parity, abort_flag, &g_status_mla, site);
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

// ===========================================================================
// Decode kernel (both dot modes).
//
// Work unit = 2 CTAs, each owning one 256-wide dv slice.  The shared-memory
// ring (5 stages; 3 with two-term dots) carries, in one order that every role
// walks, three Q slots at the start of each segment (the segment's quantised
// Q: two latent halves and the RoPE part) followed by the segment's KV pages,
// so no separate Q buffer competes with the KV pages for shared memory.
// TMEM: O 256 + two S buffers of 64 + Q latent 128 columns.
//
// 16-bit dots run as two-term E4M3 dots: Q's latent part and P each enter as
// hi + lo (hi = E4M3(x), lo = E4M3(x - hi), about bf16's 8 significant bits)
// against the cache's own E4M3 K and V codes, so no page is converted and the
// MMAs stay f8f6f4: Q.K^T takes 16 more MMAs (Q_lo from shared memory) and
// P.V 2 more (P_lo).  Q_lo is formed from the bf16 Q by the softmax warps
// when they copy the segment's Q.
// ===========================================================================
namespace f8 {
// Test hook of the bounded waits (0 = off); set by mla_set_wait_test.
__device__ int g_fault_page = 0;
constexpr int kThreads = 384;
constexpr int kOffRope8 = 4 * kLatBox;             // 64 tokens x 64 E4M3 RoPE bytes, no swizzle
constexpr int kStageBytes = kOffRope8 + kPage * 64;
constexpr int kCvtBytes = kLatBox;
constexpr int kQLoBlock = kRows * 128;             // one 128-byte column block of Q_lo (16 KB)
// Shared memory: the ring, then two buffers for a page's RoPE part as f16
// (64 keys x 128 B, 128-byte swizzle), Q's RoPE part (128 rows x 128 B f16,
// 128-byte swizzle), and P (128 rows x 64 E4M3 keys) as 8-row x 16-byte core
// matrices: row group g and 16-byte key chunk c at g * kPSbo + c * kPLbo.
// Two-term dots add P_lo (P's layout) and Q_lo: 128 rows x 512 E4M3 as four
// column blocks of kQLoBlock, each 128-byte swizzled (the K page's layout).
template <bool kTwoTerm, bool kRowScales = false>
struct Layout {
  // per-row scales give up a stage for the partner-maximum exchange (PairExchange)
  static constexpr int kStages = kTwoTerm ? 3 : (kRowScales ? 4 : 5);
  static constexpr int kOffCvt = kStages * kStageBytes;
  static constexpr int kOffQRope = kOffCvt + 2 * kCvtBytes;
  static constexpr int kOffP = kOffQRope + kRows * 128;
  static constexpr int kOffPLo = kOffP + kRows * kPage;
  static constexpr int kOffQLo = kOffPLo + (kTwoTerm ? kRows * kPage : 0);
  static constexpr int kSmemData = kOffQLo + (kTwoTerm ? 4 * kQLoBlock : 0);
  static_assert(kOffCvt % 1024 == 0 && kOffQRope % 1024 == 0 && kOffP % 1024 == 0 && kOffPLo % 1024 == 0 &&
                    kOffQLo % 1024 == 0,
                "1 KB aligned tiles");
};
constexpr int kPLbo = 128, kPSbo = 512;
constexpr float kPScale = 64.0f, kPLog2 = 6.0f;  // P is stored as E4M3(64 p)
constexpr float kTau = 2.75f;                     // 64 * 2^2.75 = 430.5 < 448
// TMEM columns: O slice, two S buffers (pages alternate), Q latent (E4M3; Q_hi with two-term dots).
constexpr uint32_t kTO = 0, kTS = 256, kTQ = 384;
// Quantised Q of a sequence, as three ring slots: slot h (h = 0, 1) holds per
// row latent bytes [256 h, 256 h + 256) at a 272-byte pitch, slot 2 the RoPE
// values as f16 at a 144-byte pitch (pitches chosen so a quarter-warp's
// 16-byte row accesses hit distinct banks).
constexpr int kQLatPitch = 272;
constexpr int kQRopePitch = 144;
constexpr int kQLatSlotBytes = kRows * kQLatPitch;
constexpr int kQRopeSlotBytes = kRows * kQRopePitch;
static_assert(kQLatSlotBytes <= kStageBytes && kQRopeSlotBytes <= kStageBytes, "a Q slot fits one stage");
static_assert(2 * kQLatSlotBytes + kQRopeSlotBytes == kMlaQBytes, "quantised-Q layout");
static_assert(kStageBytes % 1024 == 0, "1 KB aligned stages");
static_assert(kStageBytes == static_cast<int>(kPageTxBytes), "a page fills one stage");

// Per-row scales: the two threads of a query row (warps w and w + 4) swap the
// maximum of their half of a page's scaled scores instead of each scaling the
// other half too.
template <bool kOn>
struct PairExchange {};
template <>
struct PairExchange<true> {
  uint64_t pair[4];         // per row block: both warps of a row block published their half's maximum
  float pmax[2][2][kRows];  // by page parity, half, row
};

template <int kStages, bool kPair = false>
struct Bars : PairExchange<kPair> {
  uint64_t kv_full[kStages];    // stage holds its page (TMA bytes) or its Q slot (Q warps' arrival)
  uint64_t kv_empty[kStages];   // stage may be refilled
  uint64_t cvt_ready[kStages];  // the page's RoPE part is converted and its dead rows zeroed
  uint64_t s_full[2];           // S buffer b holds a page's scores
  uint64_t p_full;              // P written (one arrival per softmax warp)
  uint64_t pv_done;             // the P.V that read P completed
  uint64_t q_full, final_mma, xchg;
  uint32_t tmem_base, abort_flag, cvt_ok;
  float xsum[2][kRows];         // row-sum halves
  // per-row scales (kv_rows): by stage, the page's 64 scales sigma as bulk-copied, then (written by
  // the converter warps, one key each) sigma, log2 sigma and 1 / sigma
  alignas(16) float scl[kStages][3][kPage];
};

template <bool kTwoTerm, bool kRowScales = false>
constexpr size_t smem_bytes() {
  return Layout<kTwoTerm, kRowScales>::kSmemData + sizeof(Bars<Layout<kTwoTerm, kRowScales>::kStages, kRowScales>) +
         1024;
}
static_assert(smem_bytes<false>() <= 232448 && smem_bytes<true>() <= 232448 && smem_bytes<false, true>() <= 232448,
              "fits the 227 KB opt-in shared memory of a CTA");

// Quantises the Q rows of sequence b into the three Q slots: latent -> E4M3(q / qs),
// RoPE -> f16(q / qs), qs = smallest power of two with amax <= 448 qs.  kTpr
// threads share a row; thread `part` takes the 8-value chunks c = part (mod kTpr)
// of the row's 72 (64 latent, 8 RoPE).
template <int kTpr>
__device__ __forceinline__ void fill_q_row(const MlaParams& prm, int b, int r, int part, uint8_t* slot0,
                                           uint8_t* slot1, uint8_t* slot2, float* qs_out) {
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
  fill_q_row<8>(prm, b, r, threadIdx.x % 8, q, q + kQLatSlotBytes, q + 2 * kQLatSlotBytes,
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

// kRowScales: per-row KV scales (prm.kv_rows) instead of the per-tensor kv_scale.
// kTwoTerm: 16-bit dots as two-term E4M3 dots (per-tensor kv_scale only).
template <bool kRowScales, bool kTwoTerm>
__global__ void __launch_bounds__(f8::kThreads, 1)
    mla_fp8_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_rope,
                   const MlaParams prm) {
  static_assert(!(kRowScales && kTwoTerm), "per-row scales run with FP8 dots only");
  using namespace f8;
  using L = Layout<kTwoTerm, kRowScales>;
  constexpr int kStages = L::kStages;
  constexpr int kOffCvt = L::kOffCvt, kOffQRope = L::kOffQRope, kOffP = L::kOffP;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  Bars<kStages, kRowScales>* bars = reinterpret_cast<Bars<kStages, kRowScales>*>(smem + L::kSmemData);
  volatile uint32_t* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int unit = blockIdx.x / 2;
  const int part = blockIdx.x % 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
      mbar_init(&bars->cvt_ready[s], 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&bars->s_full[b], 1);
    mbar_init(&bars->p_full, kSoftmaxThreads / 32);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->q_full, kSoftmaxThreads / 32);
    mbar_init(&bars->final_mma, 1);
    mbar_init(&bars->xchg, kSoftmaxThreads / 32);
    if constexpr (kRowScales)
      for (int w4 = 0; w4 < 4; ++w4) mbar_init(&bars->pair[w4], 2);
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

  // Ring protocol.  Every role walks the same slot sequence: three Q slots at
  // the start of each segment (its quantised Q, prepared by mla_qprep_kernel)
  // and then its pages.  Each stage barrier completes one
  // phase per occupancy of its stage, and every role that waits on one
  // observes each of its phases in turn, so a parity wait can never pass on a
  // phase two behind or two ahead: kv_empty is waited by the producer only;
  // kv_full by the converter for every occupancy, by the MMA warp for pages
  // and by the softmax warps for Q slots; each stage is released only after
  // the converter's cvt_ready for that occupancy.
  if (warp == 0) {
    // ------------------------------------------------ TMA producer ----
    // The warp loads 32 block-table entries at a time (one per lane); lane 0
    // issues the loads.
    if (lane == 0) {
      tma_prefetch_desc(&tm_lat);
      tma_prefetch_desc(&tm_rope);
    }
    const uint64_t kv_policy = l2_evict_first_policy();
    // bounded-wait test hook: CTA 0 of unit 0 never loads its page (g_fault_page - 1) of the unit
    const int fault = (unit == 0 && part == 0) ? *reinterpret_cast<volatile int*>(&g_fault_page) : 0;
    int upg = 0;  // the unit's pages so far
    SegmentWalker walk(prm, unit);
    Segment sg;
    int k = 0;
    uint32_t issued = 0, par = 0;  // per stage: last occupant was loaded here, and its use parity
    bool ok = true;
    while (ok && walk.next(sg)) {
      // the segment's quantised Q: two latent halves and the RoPE part
      for (int q = 0; q < 3 && ok; ++q, ++k) {
        const int st = k % kStages, use = k / kStages;
        const uint32_t bytes = (q < 2) ? kQLatSlotBytes : kQRopeSlotBytes;
        bool waited = true;
        if (lane == 0) {
          waited = use == 0 || wait_bounded(&bars->kv_empty[st], (use - 1) & 1, abort_flag, &g_status_mla, __LINE__);
          if (waited) {
            mbar_arrive_expect_tx(&bars->kv_full[st], bytes);
            bulk_load(smem + st * kStageBytes,
                      prm.qbuf + static_cast<size_t>(sg.b) * kMlaQBytes + static_cast<size_t>(q) * kQLatSlotBytes,
                      bytes, &bars->kv_full[st]);
            issued |= 1u << st;
            par = (par & ~(1u << st)) | (static_cast<uint32_t>(use & 1) << st);
          }
        }
        ok = __shfl_sync(0xffffffffu, waited ? 1 : 0, 0) != 0;
      }
      if (!ok) break;
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
        for (int j = 0; j < cnt; ++j, ++k, ++upg) {
          const int phys = __shfl_sync(0xffffffffu, mine, j);
          const int st = k % kStages;
          const int use = k / kStages;
          bool waited = true;
          if (lane == 0) {
            waited = use == 0 || wait_bounded(&bars->kv_empty[st], (use - 1) & 1, abort_flag, &g_status_mla, __LINE__);
            if (waited && fault != upg + 1) {
              uint8_t* sb = smem + st * kStageBytes;
              mbar_arrive_expect_tx(&bars->kv_full[st], kPageTxBytes + (kRowScales ? kPage * 4u : 0u));
#pragma unroll
              // pages are streamed once (the unit's other CTA reads them at about the same time): evict
              // them first, keeping Q, the quantised Q and the split partials in L2 for the other kernels
#pragma unroll
              for (int q = 0; q < 4; ++q)
                tma_load_3d_hint(sb + q * kLatBox, &tm_lat, &bars->kv_full[st], q * 128, 0, phys, kv_policy);
              tma_load_3d_hint(sb + kOffRope8, &tm_rope, &bars->kv_full[st], kDLat, 0, phys, kv_policy);
              if constexpr (kRowScales)  // the page's 64 row scales (256 bytes)
                bulk_load(&bars->scl[st][0][0], prm.kv_rows + static_cast<size_t>(phys) * kPage, kPage * 4u,
                          &bars->kv_full[st]);
              issued |= 1u << st;
              par = (par & ~(1u << st)) | (static_cast<uint32_t>(use & 1) << st);
            }
          }
          if (!__shfl_sync(0xffffffffu, waited ? 1 : 0, 0)) {
            ok = false;
            break;
          }
        }
      }
    }
    // Never leave with copies in flight: wait for the last load of each stage.
    if (lane == 0)
      for (int s = 0; s < kStages; ++s)
        if ((issued >> s) & 1u) wait_bounded(&bars->kv_full[s], (par >> s) & 1u, nullptr, &g_status_mla, __LINE__);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer ----
    // The whole warp runs the loop (so descriptors stay warp-uniform) and one
    // elected lane issues -- from a lone thread each MMA costs about twice as
    // long to issue.  Pages alternate between two S buffers, so the Q.K^T of
    // page i runs while the softmax warps work on page i - 1.  Per page i: wait
    // until S buffer i % 2 was read out (page i - 2), Q.K^T as 16 E4M3 MMAs
    // (latent, Q from TMEM, K = 32) and 4 f16 MMAs (RoPE, Q from shared
    // memory, K = 16), then the P.V of page i - 1 (2 E4M3 MMAs, K = 32 keys,
    // N = 256) once its P is written.  Two-term dots add 16 Q_lo MMAs to each
    // Q.K^T and 2 P_lo MMAs to each P.V.
    {
      constexpr uint32_t idesc8 = make_idesc(0, 0, 0, 0, 64, 128);    // e4m3 x e4m3, both K-major, N = 64
      constexpr uint32_t idesc16 = make_idesc(0, 0, 0, 0, 64, 128);   // f16 x f16 (E4M3 keys are exact in f16)
      constexpr uint32_t idesc_pv = make_idesc(0, 0, 0, 1, 256, 128); // e4m3, B MN-major, N = 256
      const uint32_t t_o = tmem + kTO;
      const bool leader = elect_one();
      const uint64_t qd = make_sdesc(smem_u32(smem + kOffQRope), 16, 1024, SWIZZLE_128B);
      const uint64_t pd = make_sdesc(smem_u32(smem + kOffP), kPLbo, kPSbo, SWIZZLE_NONE);
      const uint64_t pd_lo = make_sdesc(smem_u32(smem + L::kOffPLo), kPLbo, kPSbo, SWIZZLE_NONE);
      const uint64_t qlo_d = make_sdesc(smem_u32(smem + L::kOffQLo), 16, 1024, SWIZZLE_128B);
      SegmentWalker walk(prm, unit);
      Segment sg;
      int i = 0, k = 0, seg = 0;
      int j = 0;           // next page whose P.V is due (pages j .. i - 1 have their Q.K^T issued)
      uint32_t pend = 0;   // per pending page p, byte p % 4: its stage | first-of-segment << 3
      bool ok = true;
      // the P.V of page j, once its P is written; it releases the page's stage
      auto issue_pv = [&]() -> bool {
        if (!warp_spin(&bars->p_full, j & 1, abort_flag, __LINE__)) return false;
        tc_fence_after();
        const uint32_t e = (pend >> (8 * (j & 3))) & 0xFFu;
        const int st = static_cast<int>(e & 7u);
        const bool first = ((e >> 3) & 1u) != 0;
        const uint32_t v_base = smem_u32(smem + st * kStageBytes) + part * 2 * kLatBox;
        const uint64_t vd = make_sdesc(v_base, kLatBox, 1024, SWIZZLE_128B);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          mma_f8_ss_if(leader, t_o, pd + ((kk * 2 * kPLbo) >> 4), vd + ((kk * 4096) >> 4), idesc_pv,
                       (first && kk == 0) ? 0u : 1u);
        if constexpr (kTwoTerm) {  // + P_lo . V
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma_f8_ss_if(leader, t_o, pd_lo + ((kk * 2 * kPLbo) >> 4), vd + ((kk * 4096) >> 4), idesc_pv, 1u);
        }
        tc_commit_if(leader, &bars->pv_done);
        tc_commit_if(leader, &bars->kv_empty[st]);
        ++j;
        return true;
      };
      while (ok && walk.next(sg)) {
        // The previous segment's last P.V comes first: the softmax warps write
        // its P before they copy this segment's Q.
        while (ok && j < i) ok = issue_pv();
        // the softmax warps have copied the Q slots (and the converter has seen them)
        bool qok = ok && warp_wait(&bars->q_full, seg & 1, abort_flag, __LINE__);
        for (int q = 0; q < 3 && qok; ++q)
          qok = warp_wait(&bars->cvt_ready[(k + q) % kStages], ((k + q) / kStages) & 1, abort_flag, __LINE__);
        if (!qok) {
          ok = false;
          break;
        }
        if (leader)
          for (int q = 0; q < 3; ++q) mbar_arrive(&bars->kv_empty[(k + q) % kStages]);
        __syncwarp();
        k += 3;
        // Page i's conversion is waited for while the P.V of page i - 2 runs (so
        // that Q.K^T(i) follows that P.V in the tensor pipe without a gap).  S
        // buffer i % 2 last held page i - 2, whose P (written after its S was
        // read) that P.V waited for -- or the previous segment's flush did.
        if (!warp_spin(&bars->cvt_ready[k % kStages], (k / kStages) & 1, abort_flag, __LINE__)) {
          ok = false;
          break;
        }
        for (int pg = sg.lo; pg < sg.hi; ++pg, ++i, ++k) {
          const int st = k % kStages;
          const int sbuf = i & 1;
          tc_fence_after();
          const uint32_t t_s = tmem + kTS + sbuf * kPage;
          const uint64_t kd = make_sdesc(smem_u32(smem + st * kStageBytes), 16, 1024, SWIZZLE_128B);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            mma_f8_ts_if(leader, t_s, tmem + kTQ + kk * 8, kd + ((((kk >> 2) * kLatBox) + (kk & 3) * 32) >> 4),
                         idesc8, kk > 0 ? 1u : 0u);
          if constexpr (kTwoTerm) {  // + Q_lo . K^T, Q_lo from shared memory
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              mma_f8_ss_if(leader, t_s, qlo_d + ((((kk >> 2) * kQLoBlock) + (kk & 3) * 32) >> 4),
                           kd + ((((kk >> 2) * kLatBox) + (kk & 3) * 32) >> 4), idesc8, 1u);
          }
          const uint64_t rd = make_sdesc(smem_u32(smem + kOffCvt + sbuf * kCvtBytes), 16, 1024, SWIZZLE_128B);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16_ss_if(leader, t_s, qd + ((kk * 32) >> 4), rd + ((kk * 32) >> 4), idesc16, 1u);
          tc_commit_if(leader, &bars->s_full[sbuf]);
          const uint32_t e = static_cast<uint32_t>(st) | ((pg == sg.lo) ? 8u : 0u);
          pend = (pend & ~(0xFFu << (8 * (i & 3)))) | (e << (8 * (i & 3)));
          // the P.V of the previous page (queued right behind this Q.K^T), then
          // the next page's conversion while that P.V runs
          if (pg > sg.lo && !issue_pv()) {  // j == i - 1 here
            ok = false;
            break;
          }
          if (pg + 1 < sg.hi &&
              !warp_spin(&bars->cvt_ready[(k + 1) % kStages], ((k + 1) / kStages) & 1, abort_flag, __LINE__)) {
            ok = false;
            break;
          }
        }
        ++seg;
      }
      while (ok && j < i) ok = issue_pv();  // the last P.V
      if (leader) tc_commit(&bars->final_mma);
      __syncwarp();
      warp_wait(&bars->final_mma, 0, nullptr, __LINE__);
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------- RoPE conversion, tail zeroing (64 threads) ----
    const int t = threadIdx.x - 64;  // token row of the page
    SegmentWalker walk(prm, unit);
    Segment sg;
    int k = 0, i = 0;  // ring slots, pages
    bool ok = true;
    while (ok && walk.next(sg)) {
      // the Q slots need no conversion, but their fills are waited for and
      // acknowledged like the pages' so that each stage phase is seen in turn
      if (t == 0) {
        bool filled = true;
        for (int q = 0; q < 3 && filled; ++q)
          filled = wait_bounded(&bars->kv_full[(k + q) % kStages], ((k + q) / kStages) & 1, abort_flag,
                                &g_status_mla, __LINE__);
        if (filled)
          for (int q = 0; q < 3; ++q) mbar_arrive(&bars->cvt_ready[(k + q) % kStages]);
        bars->cvt_ok = filled ? 1u : 0u;
      }
      named_bar_sync(1, 64);
      if (!bars->cvt_ok) break;
      named_bar_sync(1, 64);  // cvt_ok is rewritten below
      k += 3;
      for (int pg = sg.lo; pg < sg.hi; ++pg, ++k, ++i) {
        const int st = k % kStages;
        const int use = k / kStages;
        // conversion buffer i % 2 is free once the Q.K^T of page i - 2 completed
        if (t == 0)
          bars->cvt_ok = (wait_bounded(&bars->kv_full[st], use & 1, abort_flag, &g_status_mla, __LINE__) &&
                          (i < 2 || wait_bounded(&bars->s_full[i & 1], ((i - 2) >> 1) & 1, abort_flag, &g_status_mla, __LINE__)))
                             ? 1u
                             : 0u;
        named_bar_sync(1, 64);
        if (!bars->cvt_ok) {
          ok = false;
          break;
        }
        uint8_t* sb = smem + st * kStageBytes;
        const bool dead = (pg == sg.n - 1) && (t >= sg.s_k - pg * kPage);  // slot past the sequence end
        if constexpr (kRowScales) {  // key t's scale (1 past the end), its log2 and its inverse, for the softmax
          const float sgm = dead ? 1.f : bars->scl[st][0][t];
          bars->scl[st][0][t] = sgm;
          bars->scl[st][1][t] = lg2_approx(sgm);
          bars->scl[st][2][t] = 1.f / sgm;
        }
        const uint4 z = make_uint4(0, 0, 0, 0);
        const int sw = t & 7;
        const uint4* src = reinterpret_cast<const uint4*>(sb + kOffRope8 + t * 64);
        uint8_t* dst = smem + kOffCvt + (i & 1) * kCvtBytes + t * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 lo = z, hi = z;
          if (!dead) {
            const uint4 v = src[c];
            lo.x = e4m3x2_to_f16x2(v.x & 0xFFFFu);
            lo.y = e4m3x2_to_f16x2(v.x >> 16);
            lo.z = e4m3x2_to_f16x2(v.y & 0xFFFFu);
            lo.w = e4m3x2_to_f16x2(v.y >> 16);
            hi.x = e4m3x2_to_f16x2(v.z & 0xFFFFu);
            hi.y = e4m3x2_to_f16x2(v.z >> 16);
            hi.z = e4m3x2_to_f16x2(v.w & 0xFFFFu);
            hi.w = e4m3x2_to_f16x2(v.w >> 16);
          }
          *reinterpret_cast<uint4*>(dst + (((2 * c) ^ sw) << 4)) = lo;
          *reinterpret_cast<uint4*>(dst + (((2 * c + 1) ^ sw) << 4)) = hi;
        }
        if (dead) {  // zero the slot's V row (all four 128-byte slices)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4* row = reinterpret_cast<uint4*>(sb + j * kLatBox + t * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) row[c] = z;
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 64);
        if (t == 0) mbar_arrive(&bars->cvt_ready[st]);
      }
    }
  } else {
    // ------------------ softmax / Q copy / epilogue (8 warps, 2 per row) ----
    const int hf = (warp - 4) / 4;         // which half of the row
    const int r = (warp % 4) * 32 + lane;  // query row = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    const float kv_scale = kRowScales ? 1.f : *prm.kv_scale;  // per-row scales enter through P and S
    const int R = prm.s_q * prm.h_q;
    constexpr int kOHalf = 128;  // O columns of this thread
    uint32_t xphase = 0;
    auto xsync = [&]() -> bool {  // bounded, abort-aware exchange point of the 256 softmax threads
      warp_arrive(&bars->xchg);
      const bool ok = warp_wait(&bars->xchg, xphase & 1, abort_flag, __LINE__);
      ++xphase;
      return ok;
    };
    // Copies this half of the Q row of the segment whose Q slots start at ring
    // slot kq: latent bytes [256 hf, +256) into TMEM columns kTQ + 64 hf..,
    // RoPE values [32 hf, +32) into the shared Q RoPE tile (128-byte swizzle).
    auto copy_q = [&](int kq, int b_seq, float& qs_out) -> bool {
      const int st = (kq + hf) % kStages, use = (kq + hf) / kStages;
      const int st_r = (kq + 2) % kStages, use_r = (kq + 2) / kStages;
      if (!warp_wait(&bars->kv_full[st], use & 1, abort_flag, __LINE__) ||
          !warp_wait(&bars->kv_full[st_r], use_r & 1, abort_flag, __LINE__))
        return false;
      const uint4* lat = reinterpret_cast<const uint4*>(smem + st * kStageBytes + r * kQLatPitch);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = lat[4 * ch + c];
          pk[4 * c + 0] = v.x;
          pk[4 * c + 1] = v.y;
          pk[4 * c + 2] = v.z;
          pk[4 * c + 3] = v.w;
        }
        tmem_st16(lane_base + kTQ + (4 * hf + ch) * 16, pk);
      }
      {
        const uint4* rope = reinterpret_cast<const uint4*>(smem + st_r * kStageBytes + r * kQRopePitch);
        uint8_t* dst = smem + kOffQRope + r * 128;
#pragma unroll
        for (int c = 4 * hf; c < 4 * hf + 4; ++c) *reinterpret_cast<uint4*>(dst + ((c ^ (r & 7)) << 4)) = rope[c];
      }
      qs_out = prm.qscale[static_cast<size_t>(b_seq) * kRows + r];
      if constexpr (kTwoTerm) {
        // Q_lo = E4M3(x - E4M3(x)), x = q / qs, for this half's latent bytes [256 hf, +256) of the
        // row, from the bf16 Q (the hi term recomputed with the prep kernel's rounding), into
        // column block x / 128 of the 128-byte-swizzled Q_lo tile; rows past R stay zero
        const float inv_qs = __uint_as_float((254u << 23) - __float_as_uint(qs_out));  // 1 / qs, a power of two
        const bool live = r < R;
        const uint4* qg =
            reinterpret_cast<const uint4*>(prm.q + (static_cast<size_t>(b_seq) * R + (live ? r : 0)) * kD) + 32 * hf;
        uint8_t* qlo = smem + L::kOffQLo + r * 128;
#pragma unroll 4
        for (int c = 0; c < 16; ++c) {  // 16 values = one 16-byte chunk of Q_lo
          const uint4 a = live ? __ldg(qg + 2 * c) : make_uint4(0, 0, 0, 0);
          const uint4 d = live ? __ldg(qg + 2 * c + 1) : make_uint4(0, 0, 0, 0);
          uint32_t hi, lo[4];
          split_e4m3x4(bf16_lo(a.x) * inv_qs, bf16_hi(a.x) * inv_qs, bf16_lo(a.y) * inv_qs, bf16_hi(a.y) * inv_qs,
                       hi, lo[0]);
          split_e4m3x4(bf16_lo(a.z) * inv_qs, bf16_hi(a.z) * inv_qs, bf16_lo(a.w) * inv_qs, bf16_hi(a.w) * inv_qs,
                       hi, lo[1]);
          split_e4m3x4(bf16_lo(d.x) * inv_qs, bf16_hi(d.x) * inv_qs, bf16_lo(d.y) * inv_qs, bf16_hi(d.y) * inv_qs,
                       hi, lo[2]);
          split_e4m3x4(bf16_lo(d.z) * inv_qs, bf16_hi(d.z) * inv_qs, bf16_lo(d.w) * inv_qs, bf16_hi(d.w) * inv_qs,
                       hi, lo[3]);
          const int x = 256 * hf + 16 * c;
          *reinterpret_cast<uint4*>(qlo + (x >> 7) * kQLoBlock + ((((x & 127) >> 4) ^ (r & 7)) << 4)) =
              make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      fence_proxy_async_smem();  // the Q RoPE (and Q_lo) tiles are read by the MMAs, the slots refilled by TMA
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(&bars->q_full);
      return true;
    };

    SegmentWalker walk(prm, unit);
    Segment sg;
    int i = 0, k = 0, seg = 0;
    float qs_next = 1.f;
    bool ok = walk.next(sg) && copy_q(0, sg.b, qs_next);
    while (ok) {
      const float qs = qs_next;
      const float c_row = prm.softmax_scale * kLog2e * qs * kv_scale;
      SegmentWalker peek = walk;
      Segment nx;
      const bool has_next = peek.next(nx);
      const int k_next = k + 3 + (sg.hi - sg.lo);
      const int col0 = part * 256 + hf * kOHalf;  // this thread's O columns
      // keys visible to this row (bottom-right causal alignment); pages wholly
      // below every row's limit need no mask
      const int qtok = (r < R) ? r / prm.h_q : 0;
      const int visible = prm.causal ? (sg.s_k - prm.s_q + qtok + 1) : sg.s_k;
      const int min_visible = prm.causal ? (sg.s_k - prm.s_q + 1) : sg.s_k;
      float m_run = kNegInf, l_run = 0.f;  // l_run sums the stored-scale p (kPScale p)
      for (int pg = sg.lo; pg < sg.hi; ++pg, ++i) {
        const int sbuf = i & 1;
        if (!warp_spin(&bars->s_full[sbuf], (i >> 1) & 1, abort_flag, __LINE__)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // Both halves of the row are read: the other half only for the row max,
        // so each warp takes the max of all 64 keys without waiting on its partner.
        uint32_t s[32], so[kRowScales ? 1 : 32];
        tmem_ld32(lane_base + kTS + sbuf * kPage + 32 * hf, s);
        if constexpr (!kRowScales) tmem_ld32(lane_base + kTS + sbuf * kPage + 32 * (1 - hf), so);
        // per-row scales: the page's stage (its slot follows the segment's three Q slots); its
        // conversion barrier covers the scale arrays, and its phase is this page's (the stage is
        // refilled only after this page's P.V)
        const int pslot = k + 3 + (pg - sg.lo);
        const int pst = pslot % kStages;
        if constexpr (kRowScales) {
          if (!warp_spin(&bars->cvt_ready[pst], (pslot / kStages) & 1, abort_flag, __LINE__)) {
            ok = false;
            break;
          }
        }
        tmem_ld_wait();

        if (pg * kPage + kPage > min_visible) {
          const int base = pg * kPage + 32 * hf, base_o = pg * kPage + 32 * (1 - hf);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (base + c >= visible) s[c] = __float_as_uint(kNegInf);
            if constexpr (!kRowScales)
              if (base_o + c >= visible) so[c] = __float_as_uint(kNegInf);
          }
        }
        float mx;
        if constexpr (kRowScales) {
          // u_j = s_j c sigma_j + log2 sigma_j: the key's score with its K scale, plus its V scale's
          // log, so that P' = 2^(u_j - m) carries sigma_j (masked keys stay -inf)
          // (16-byte loads: the same four keys' scales for every row of the warp)
          const float4* sg4 = reinterpret_cast<const float4*>(bars->scl[pst][0]);
          const float4* lg4 = reinterpret_cast<const float4*>(bars->scl[pst][1]);
          auto scale4 = [&](uint32_t* v, float4 g, float4 l) {
            v[0] = __float_as_uint(fmaf(__uint_as_float(v[0]), c_row * g.x, l.x));
            v[1] = __float_as_uint(fmaf(__uint_as_float(v[1]), c_row * g.y, l.y));
            v[2] = __float_as_uint(fmaf(__uint_as_float(v[2]), c_row * g.z, l.z));
            v[3] = __float_as_uint(fmaf(__uint_as_float(v[3]), c_row * g.w, l.w));
          };
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) scale4(s + 4 * c4, sg4[8 * hf + c4], lg4[8 * hf + c4]);
          // this half's maximum, swapped with the row's other thread (warp w + 4 or w - 4) through the
          // pair barrier; both then take the same row maximum
          float m11[11];
#pragma unroll
          for (int c = 0; c < 10; ++c)
            m11[c] = fmax3(__uint_as_float(s[3 * c]), __uint_as_float(s[3 * c + 1]), __uint_as_float(s[3 * c + 2]));
          m11[10] = fmaxf(__uint_as_float(s[30]), __uint_as_float(s[31]));
          const float m_own = fmax3(fmax3(m11[0], m11[1], m11[2]), fmax3(m11[3], m11[4], m11[5]),
                                    fmax3(fmax3(m11[6], m11[7], m11[8]), m11[9], m11[10]));
          bars->pmax[i & 1][hf][r] = m_own;
          warp_arrive(&bars->pair[warp % 4]);
          if (!warp_spin(&bars->pair[warp % 4], i & 1, abort_flag, __LINE__)) {
            ok = false;
            break;
          }
          mx = fmaxf(m_own, bars->pmax[i & 1][1 - hf][r]);
        } else {
          // row max of the 64 scores as a tree of three-way maxima
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
          const float m3a = fmax3(m8[0], m8[1], m8[2]), m3b = fmax3(m8[3], m8[4], m8[5]);
          mx = fmax3(m3a, m3b, fmaxf(m8[6], m8[7])) * c_row;  // c_row > 0; both warps agree
        }
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_run + kTau) {
          alpha = ex2_approx(m_run - mx);
          rescale = (pg != sg.lo);
          m_run = mx;
        }
        const float bias = (m_run == kNegInf) ? 0.f : (kPLog2 - m_run);
        float sum = 0.f;
        uint32_t pk[8], pk_lo[kTwoTerm ? 8 : 1];
        if constexpr (kRowScales) {
          // P' = 2^(u_j - m) (stored, times kPScale); the row sum takes P' / sigma_j = 2^(s_j c sigma_j - m)
          const float4* iv4 = reinterpret_cast<const float4*>(bars->scl[pst][2] + 32 * hf);
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float p0 = ex2_approx(__uint_as_float(s[c]) + bias);
            const float p1 = ex2_approx(__uint_as_float(s[c + 1]) + bias);
            const float p2 = ex2_approx(__uint_as_float(s[c + 2]) + bias);
            const float p3 = ex2_approx(__uint_as_float(s[c + 3]) + bias);
            const float4 iv = iv4[c / 4];
            sum = fmaf(p3, iv.w, fmaf(p2, iv.z, fmaf(p1, iv.y, fmaf(p0, iv.x, sum))));
            pk[c / 4] = pack_e4m3x4(p0, p1, p2, p3);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(s[c]), c_row, bias));
            const float p1 = ex2_approx(fmaf(__uint_as_float(s[c + 1]), c_row, bias));
            const float p2 = ex2_approx(fmaf(__uint_as_float(s[c + 2]), c_row, bias));
            const float p3 = ex2_approx(fmaf(__uint_as_float(s[c + 3]), c_row, bias));
            sum += (p0 + p1) + (p2 + p3);
            if constexpr (kTwoTerm)
              split_e4m3x4(p0, p1, p2, p3, pk[c / 4], pk_lo[c / 4]);
            else
              pk[c / 4] = pack_e4m3x4(p0, p1, p2, p3);
          }
        }
        l_run = l_run * alpha + sum;

        // P has one tile and O one accumulator: the previous page's P.V must
        // have completed before either is touched
        if (i >= 1 && !warp_spin(&bars->pv_done, (i - 1) & 1, abort_flag, __LINE__)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
          const float f = rescale ? alpha : 1.f;
#pragma unroll 1
          for (int ch = 0; ch < kOHalf / 32; ++ch) {
            const uint32_t col = kTO + hf * kOHalf + ch * 32;
            uint32_t o[32];
            tmem_ld32(lane_base + col, o);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
            tmem_st32(lane_base + col, o);
          }
          tmem_st_wait();
        }
        {  // this warp's 32 keys of row r: 16-byte chunks 2 hf and 2 hf + 1
          uint8_t* prow = smem + kOffP + (r >> 3) * kPSbo + (r & 7) * 16;
          *reinterpret_cast<uint4*>(prow + (2 * hf) * kPLbo) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(prow + (2 * hf + 1) * kPLbo) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          if constexpr (kTwoTerm) {  // P_lo, same layout
            uint8_t* plo = prow + (L::kOffPLo - kOffP);
            *reinterpret_cast<uint4*>(plo + (2 * hf) * kPLbo) = make_uint4(pk_lo[0], pk_lo[1], pk_lo[2], pk_lo[3]);
            *reinterpret_cast<uint4*>(plo + (2 * hf + 1) * kPLbo) = make_uint4(pk_lo[4], pk_lo[5], pk_lo[6], pk_lo[7]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(&bars->p_full);
        // the segment's last Q.K^T is done: the next segment's Q may replace it now
        if (pg == sg.hi - 1 && has_next && !copy_q(k_next, nx.b, qs_next)) {
          ok = false;
          break;
        }
      }
      if (!ok) break;

      // ---- epilogue: O is final once the segment's last P.V completes ----
      bars->xsum[hf][r] = l_run;
      if (!xsync()) break;
      const float l_tot = (bars->xsum[0][r] + bars->xsum[1][r]) * (1.0f / kPScale);  // sum of p
      const bool whole = (sg.lo == 0 && sg.hi == sg.n);
      const float o_scale = kv_scale / kPScale;  // tensor-core units -> true units
      const float f = whole ? ((l_tot > 0.f) ? o_scale / l_tot : 0.f) : o_scale;
      const int slot = whole ? 0 : prm.num_splits[sg.b] + sg.split;
      if (!warp_wait(&bars->pv_done, (i - 1) & 1, abort_flag, __LINE__)) break;
      tc_fence_after();
      // O out as bf16, 32 columns at a time.  A thread holds one row; groups of
      // four lanes transpose their 16-byte pieces so that each store writes
      // 64-byte runs of rows.  A whole sequence goes straight to out, a piece
      // to its bf16 partial slot; the combine kernel adds the LSE correction.
      const int grow = (warp % 4) * 32 + (lane & ~3);  // the lane group's first row
      uint16_t* obase = whole ? prm.out + static_cast<size_t>(sg.b) * R * kDV
                              : prm.ws_o + static_cast<size_t>(slot) * kRows * kDV;
#pragma unroll 1
      for (int ch = 0; ch < kOHalf / 32; ++ch) {
        uint32_t o[32];
        tmem_ld32(lane_base + kTO + hf * kOHalf + ch * 32, o);
        tmem_ld_wait();
        uint4 pc[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          pc[c].x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * f, __uint_as_float(o[8 * c + 1]) * f);
          pc[c].y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * f, __uint_as_float(o[8 * c + 3]) * f);
          pc[c].z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * f, __uint_as_float(o[8 * c + 5]) * f);
          pc[c].w = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * f, __uint_as_float(o[8 * c + 7]) * f);
        }
        lane_group_transpose<4>(pc, lane);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          if (grow + kk < R)
            *reinterpret_cast<uint4*>(obase + static_cast<size_t>(grow + kk) * kDV + col0 + ch * 32 + 8 * (lane & 3)) =
                pc[kk];
      }
      if (r < R && part == 0 && hf == 0) {  // the row's (uncorrected) LSE, or the piece's (m, l)
        if (whole) {
          prm.lse[static_cast<size_t>(sg.b) * R + r] = (l_tot > 0.f) ? (m_run + lg2_approx(l_tot)) * kLn2 : kNegInf;
        } else {
          prm.ws_ml[static_cast<size_t>(slot) * kRows + r] = make_float2((l_tot > 0.f) ? m_run : kNegInf, l_tot);
        }
      }
      if (!has_next) break;
      walk.next(sg);
      k = k_next;
      ++seg;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool kRowScales, bool kTwoTerm>
cudaError_t launch_instance(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const MlaParams& prm,
                            int num_units, cudaStream_t stream) {
  constexpr size_t kBytes = f8::smem_bytes<kTwoTerm, kRowScales>();
  static std::atomic<uint64_t> configured{0};  // per device: CUDA keeps the limit per device
  const cudaError_t e = configure_once(configured, [] {
    return cudaFuncSetAttribute(mla_fp8_kernel<kRowScales, kTwoTerm>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kBytes));
  });
  if (e != cudaSuccess) return e;
  return launch_dependent(mla_fp8_kernel<kRowScales, kTwoTerm>, dim3(num_units * 2), dim3(f8::kThreads), kBytes,
                          stream, tm_lat, tm_rope, prm);
}

}  // namespace mla

cudaError_t launch_mla_decode_fp8(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const MlaParams& prm,
                                  int num_units, cudaStream_t stream) {
  return prm.kv_rows ? mla::launch_instance<true, false>(tm_lat, tm_rope, prm, num_units, stream)
                     : mla::launch_instance<false, false>(tm_lat, tm_rope, prm, num_units, stream);
}

cudaError_t launch_mla_decode_16bit(const CUtensorMap& tm_lat, const CUtensorMap& tm_rope, const MlaParams& prm,
                                    int num_units, cudaStream_t stream) {
  if (prm.kv_rows) return cudaErrorInvalidValue;
  return mla::launch_instance<false, true>(tm_lat, tm_rope, prm, num_units, stream);
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
