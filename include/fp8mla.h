/*
 * fp8mla.h -- C ABI of libfp8mla.so: decode-phase attention over an FP8
 * (E4M3, OCP "fn" encoding) paged KV cache on sm_103a.
 *
 * Three variants of one operation, all "softmax(scale * q . k) @ v over the
 * keys of a paged cache", plus the bookkeeping around them:
 *
 *   fp8mla_get_metadata / fp8mla_decode  -- dense MLA decode: d = 576
 *       (512 latent + 64 RoPE), dv = 512 (V is the first 512 dims of the
 *       same cached row), one shared KV head, s_q = 1..2 query tokens with a
 *       bottom-right causal mask.  FlashMLA "update fp8 support":
 *       Improvements (FP8 Q and KV, Q.K over nine 64-wide K chunks with the
 *       RoPE chunk kept at 16 bit) and the H800 test shape (b, s_q, h_q,
 *       h_kv = 1, d = 576, dv = 512, causal).
 *   sparse_mla_decode -- top-k sparse MLA: each query token attends to the
 *       rows listed in its top-k index list of one flat cache (rope-free
 *       d = dv = 512).  aiter "Support fp8 KV caches and fp8 dots in
 *       sparse_mla_fwd on gfx942": Technical details (in-kernel Q
 *       quantisation, P quantised as p * 128 with the factor divided out in
 *       the epilogue) and Results (16 heads, top-k 2048).
 *   paged_gqa_decode -- grouped-query paged decode with separate K and V
 *       caches and split-KV flash-decoding.  InfiniCore "add FP8 blockwise
 *       dequantize/GEMM operators and FP8(E4M3) KV cache support in paged
 *       attention": Summary (FP8 decode kernel, split-kv with a combine
 *       kernel, the "auto" waves heuristic) and the split-kv commit
 *       (partial (max, sum_exp, weighted sum) triples, empty shards publish
 *       m = -inf, l = 0, acc = 0).
 *
 * and the step that fills the cache:
 *
 *   fp8_paged_cache_write -- quantise new bf16 K or V rows into an E4M3
 *       paged cache, with per-row scales amax / 448 or one given per-tensor
 *       scale.  InfiniCore page, Summary: the paged_caching write kernel.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument that names a tensor is a DEVICE pointer unless
 *    stated otherwise; the caller owns all memory (inputs, outputs,
 *    workspace, metadata).  The library allocates nothing on these calls;
 *    it keeps only a small host-side cache of encoded TMA descriptors.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and returns as soon as its kernels are enqueued.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns a status and launches nothing.  Device-side problems
 *    (an index out of range, a bounded wait that ran out) never trap: the
 *    kernel records a bit in a device status word and skips the work;
 *    fp8mla_get_last_device_error() reads and clears it.
 *  - Values: the cache holds E4M3 bytes; true value = kv_scale * decode(byte)
 *    with one float32 per-tensor scale (amax / 448 on the InfiniCore page)
 *    passed as a DEVICE pointer to one float.  Q is bf16.  Outputs: bf16
 *    `out` and float32 `lse` = natural log of sum_j exp(scale * q . k_j).
 *  - A row that sees no key (empty cache, causal cut, all indices -1) gets
 *    out = 0 and lse = -inf (InfiniCore zero-length-row commit; FlashInfer
 *    "add xqa fp8 mha and fp8 kv cache", review of fully masked rows).
 *  - Cache bytes past a sequence's length and pages the block table does not
 *    reference are never read and may hold anything (NaN included).
 */
#ifndef FP8MLA_H
#define FP8MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FP8MLA_API __attribute__((visibility("default")))
#else
#define FP8MLA_API
#endif

typedef struct CUstream_st* fp8mla_stream_t; /* same type as cudaStream_t */

typedef enum {
  FP8MLA_OK = 0,
  FP8MLA_ERR_INVALID_ARG = 1,       /* null pointer, bad shape, missing kv scale, ... */
  FP8MLA_ERR_UNSUPPORTED_DTYPE = 2, /* cache encoding other than OCP E4M3 */
  FP8MLA_ERR_WORKSPACE_TOO_SMALL = 3,
  FP8MLA_ERR_CUDA = 4,              /* a CUDA runtime/driver call failed */
  FP8MLA_ERR_DEVICE = 5             /* not a launch failure: see fp8mla_get_last_device_error */
} fp8mla_status_t;

/* Precision of the two dot products (Q.K and P.V).
 *  FP8MLA_DOT_16BIT: "bf16 dots" on the aiter page: Q and P keep bf16's 8
 *    significant bits, K and V are the cache's exact E4M3 values.  Dense MLA
 *    computes them as two-term E4M3 dots: the latent part of Q (with a
 *    per-row power-of-two scale) and P (as 64 * p) each enter as hi + lo,
 *    hi = E4M3(x), lo = E4M3(x - hi); the RoPE part of Q.K is f16.
 *  FP8MLA_DOT_FP8:   the latent part of Q is quantised to E4M3 with a
 *    per-row power-of-two scale, the RoPE part of Q.K stays 16-bit (f16 in
 *    dense MLA; FlashMLA page, Improvements), and P is quantised as E4M3
 *    (64 * p in dense MLA, 128 * p in sparse MLA; aiter page, Technical
 *    details).
 *  The first-order effect of rounding Q on the LSE is corrected (dense MLA,
 *  both modes; sparse MLA). */
typedef enum { FP8MLA_DOT_16BIT = 0, FP8MLA_DOT_FP8 = 1 } fp8mla_dot_mode_t;

/* Encoding of the cache bytes.  Only FP8MLA_KV_E4M3 (OCP e4m3 "fn", or a
 * uint8 view of it) is accepted; the others are refused with
 * FP8MLA_ERR_UNSUPPORTED_DTYPE instead of being misread (aiter page,
 * Technical details: "a typed cache in the other arch's encoding is
 * refused"). */
typedef enum {
  FP8MLA_KV_E4M3 = 0,
  FP8MLA_KV_E4M3FNUZ = 1,
  FP8MLA_KV_E5M2 = 2,
  FP8MLA_KV_OTHER = 3
} fp8mla_kv_dtype_t;

/* Device status bits reported by fp8mla_get_last_device_error. */
#define FP8MLA_DEV_WAIT_TIMEOUT 0x1u   /* a bounded mbarrier wait ran out; the CTA stopped */
#define FP8MLA_DEV_BAD_PAGE 0x2u       /* block-table entry outside [0, num_pages) */
#define FP8MLA_DEV_BAD_SEQLEN 0x4u     /* seqlen < 0 or more pages than the block table row */
#define FP8MLA_DEV_BAD_INDEX 0x8u      /* top-k index outside [-1, num_tokens) */
#define FP8MLA_DEV_BAD_SLOT 0x10u      /* cache-write slot >= num_blocks * page_size */

/* ------------------------------------------------------------------ MLA ---
 * Work units.  The dense MLA kernel runs one work unit per pair of SMs (the
 * two CTAs of a unit each own one half of dv).  fp8mla_metadata_units(n)
 * is the number of units for a GPU with n SMs: max(1, n / 2). */
FP8MLA_API int fp8mla_metadata_units(int num_sms);

/* fp8mla_get_metadata -- split the batch's (sequence, 64-token page) work
 * list into `num_units` contiguous page ranges of balanced cost (each page
 * costs 1, each (sequence, unit) segment a fixed 4 more).  Computed once per
 * decode step on the device, reused by every layer.
 *   cache_seqlens  int32 [b] (device)
 *   h_q, s_q       query heads and tokens (h_q * s_q <= 128)
 *   num_units      fp8mla_metadata_units(num_sms)
 *   force_splits   0 = balanced; k > 0 = cut every sequence into min(k,
 *                  pages) near-equal chunks, one unit each (needs
 *                  b * k <= num_units) -- for split-KV tests
 *   tile_sched     int32 [num_units][8] (device, written): {b_begin,
 *                  page_begin, b_end, page_end, split index of the first
 *                  segment, 0, 0, 0}; the range ends before (b_end, page_end)
 *   num_splits     int32 [b + 1] (device, written): prefix sum of the number
 *                  of units touching each sequence (0 for an empty one). */
FP8MLA_API fp8mla_status_t fp8mla_get_metadata(const int32_t* cache_seqlens, int b, int h_q, int s_q, int num_units,
                                    int force_splits, int32_t* tile_sched, int32_t* num_splits,
                                    fp8mla_stream_t stream);

/* Workspace of fp8mla_decode: (b + num_units) split-KV partial slots of
 * 128 x 512 bf16 accumulators plus 128 (m, l) pairs each, then per sequence
 * its quantised Q, the E4M3 hi term in both dot modes (88 064 bytes: the
 * decode kernel's Q slots), and 128 Q scales. */
FP8MLA_API size_t fp8mla_workspace_bytes(int b, int s_q, int h_q, int num_units);

/* fp8mla_decode -- dense MLA decode over the paged E4M3 cache.
 *   q              bf16 [b, s_q, h_q, 576]
 *   kv_cache       E4M3 bytes [num_pages, 64, 576]; row = 512 latent || 64 RoPE
 *   kv_dtype       must be FP8MLA_KV_E4M3
 *   block_table    int32 [b, max_pages]; logical page p of sequence i lives at
 *                  physical page block_table[i * max_pages + p]
 *   cache_seqlens  int32 [b]; keys per sequence (0 allowed)
 *   kv_scale       float32 [1] (device): per-tensor dequantisation scale; NULL
 *                  is refused (InfiniCore "F8 cache without scales fails
 *                  loudly (Bad Parameter)")
 *   softmax_scale  multiplier of q . k (e.g. 1/sqrt(576))
 *   causal         1: query token i of s_q sees keys j < s_k - s_q + i + 1
 *   tile_sched, num_splits, num_units -- from fp8mla_get_metadata on the same
 *                  cache_seqlens
 *   workspace      >= fp8mla_workspace_bytes(b, s_q, h_q, num_units) bytes,
 *                  256-byte aligned; contents need not be initialised
 *   out            bf16 [b, s_q, h_q, 512] (written)
 *   lse            float32 [b, s_q, h_q] (written)
 *   dot_mode       FP8MLA_DOT_FP8 or FP8MLA_DOT_16BIT
 * Requires h_q * s_q <= 128, kv_cache / q / out 16-byte aligned. */
FP8MLA_API fp8mla_status_t fp8mla_decode(const void* q, const void* kv_cache, fp8mla_kv_dtype_t kv_dtype, int num_pages,
                              const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                              const float* kv_scale, float softmax_scale, int causal, const int32_t* tile_sched,
                              const int32_t* num_splits, int num_units, void* workspace, size_t workspace_bytes,
                              void* out, float* lse, fp8mla_dot_mode_t dot_mode, int b, int s_q, int h_q,
                              fp8mla_stream_t stream);

/* fp8mla_decode_ext -- fp8mla_decode with one dequantisation scale per cached
 * row (InfiniCore page, Summary: FP8 caches carry scales of shape
 * [num_blocks, num_kv_heads, block_size]; here one KV head, so [num_pages, 64]).
 *   kv_scale_rows  float32 [num_pages, 64] (device, 16-byte aligned) or NULL;
 *                  when set, row t of physical page p (its 512 latent and 64
 *                  RoPE values, K and V alike) is E4M3 code times
 *                  kv_scale_rows[p * 64 + t], every scale of a row a key uses
 *                  must be positive and finite, kv_scale is ignored (may be
 *                  NULL), and only FP8MLA_DOT_FP8 is accepted
 *                  (FP8MLA_ERR_INVALID_ARG otherwise)
 *   kv_scale_rows NULL: exactly fp8mla_decode.
 * Other arguments, results and errors as fp8mla_decode. */
FP8MLA_API fp8mla_status_t fp8mla_decode_ext(const void* q, const void* kv_cache, fp8mla_kv_dtype_t kv_dtype,
                                             int num_pages, const int32_t* block_table, int max_pages,
                                             const int32_t* cache_seqlens, const float* kv_scale,
                                             const float* kv_scale_rows, float softmax_scale, int causal,
                                             const int32_t* tile_sched, const int32_t* num_splits, int num_units,
                                             void* workspace, size_t workspace_bytes, void* out, float* lse,
                                             fp8mla_dot_mode_t dot_mode, int b, int s_q, int h_q,
                                             fp8mla_stream_t stream);

/* ----------------------------------------------------------- sparse MLA ---
 * sparse_mla_decode -- query token t attends to the cache rows
 * topk_idx[t][0..topk) (an index of -1 is skipped), d = dv = 512 rope-free.
 *   q            bf16 [s_q, h_q, 512], 1 <= h_q <= 16 (the heads are the N
 *                dimension of one MMA tile); h_q > 16 -> FP8MLA_ERR_INVALID_ARG
 *   kv_cache     E4M3 bytes [num_tokens, 512], num_tokens < 2^31
 *   topk_idx     int32 [s_q, topk]; an index outside [-1, num_tokens) sets
 *                FP8MLA_DEV_BAD_INDEX and the key is skipped
 *   kv_scale     float32 [1] (device), NULL refused
 *   num_splits   0 = auto (about one CTA per SM over s_q tokens, at most one
 *                split per 128-key chunk), 1 = no split-K (one pass over all
 *                keys), k > 1 = keys cut into k contiguous shards merged by
 *                the combine step
 *   workspace    >= sparse_mla_workspace_bytes(s_q, h_q, topk, num_splits)
 *                bytes, 256-byte aligned; may be NULL when that is 0
 *   out          bf16 [s_q, h_q, 512]; lse float32 [s_q, h_q]
 *   dot_mode     must be FP8MLA_DOT_FP8 (Q quantised per row with a
 *                power-of-two scale, P as E4M3(128 p)); FP8MLA_DOT_16BIT is
 *                refused with FP8MLA_ERR_INVALID_ARG (this variant runs the
 *                aiter page's FP8-dot path only) */
FP8MLA_API fp8mla_status_t sparse_mla_decode(const void* q, const void* kv_cache, fp8mla_kv_dtype_t kv_dtype,
                                  int64_t num_tokens, const int32_t* topk_idx, int topk, const float* kv_scale,
                                  float softmax_scale, int num_splits, void* workspace, size_t workspace_bytes,
                                  void* out, float* lse, fp8mla_dot_mode_t dot_mode, int s_q, int h_q,
                                  fp8mla_stream_t stream);

/* Workspace bytes of sparse_mla_decode with these arguments: the split
 * partials of the split count the call will choose (auto uses the SM count
 * of the current device); 0 when that is a single split. */
FP8MLA_API size_t sparse_mla_workspace_bytes(int s_q, int h_q, int topk, int num_splits);

/* ------------------------------------------------------------------ GQA ---
 * paged_gqa_decode -- grouped-query decode; q head h reads KV head
 * h / (h_q / h_kv).
 *   q            bf16 [bs, h_q, head_dim]
 *   k_cache      E4M3 bytes [num_blocks, h_kv, page_size, head_dim]
 *   v_cache      E4M3 bytes [num_blocks, h_kv, page_size, head_dim]
 *   k_scale, v_scale  float32 [1] each (device), NULL refused
 *   block_table  int32 [bs, max_blocks]; seqlens int32 [bs]
 *   num_splits   0 = auto: when bs * h_kv CTAs already fill the GPU, every
 *                sequence is cut into a few key shards (about six CTAs per
 *                SM, at least 8 steps of 128 keys each, at most 16) so that
 *                unequal lengths balance; otherwise the fewest shards that
 *                fill the waves; k >= 1 forced
 *   workspace    >= paged_gqa_workspace_bytes(bs, h_q, head_dim, splits)
 *   out          bf16 [bs, h_q, head_dim]; lse float32 [bs, h_q]
 * Requires head_dim == 128, page_size == 16, h_q % h_kv == 0, h_q / h_kv <= 16. */
FP8MLA_API fp8mla_status_t paged_gqa_decode(const void* q, const void* k_cache, const void* v_cache,
                                 fp8mla_kv_dtype_t kv_dtype, int num_blocks, const float* k_scale,
                                 const float* v_scale, const int32_t* block_table, int max_blocks,
                                 const int32_t* seqlens, float softmax_scale, int num_splits, void* workspace,
                                 size_t workspace_bytes, void* out, float* lse, int bs, int h_q, int h_kv,
                                 int head_dim, int page_size, fp8mla_stream_t stream);

/* paged_gqa_decode_ext -- paged_gqa_decode with per-row KV scales and the XQA
 * options (FlashInfer "add xqa fp8 mha and fp8 kv cache": launcher arguments
 * for speculative decoding, sliding window and attention sinks; InfiniCore
 * page, Summary: scales of shape [num_blocks, num_kv_heads, block_size]).
 *   q            bf16 [bs, q_len, h_q, head_dim]: q_len query tokens per
 *                sequence, taken to be its last q_len cache positions (token i
 *                at position s_k - q_len + i)
 *   k_scale, v_scale  float32 [1] each, or with scale_per_row != 0 one float
 *                per cached row, [num_blocks, h_kv, page_size], 16-byte aligned
 *   spec_mask    uint8 [bs, q_len, q_len] (device) or NULL: token i sees key
 *                s_k - q_len + c of its own block iff spec_mask[b][i][c] != 0;
 *                NULL = causal inside the block (c <= i).  Keys before the
 *                block are always visible.
 *   window       0 = off; W > 0 keeps only keys j with (s_k - q_len + i) - j < W
 *   sinks        float32 [h_q] (device) or NULL: head h's softmax denominator
 *                gains e^{sinks[h]} (a key without value; -inf = no sink)
 *   out          bf16 [bs, q_len, h_q, head_dim]; lse float32 [bs, q_len, h_q]
 * A row that sees no key gets out = 0 and lse = its sink (-inf without one).
 * Requires q_len >= 1 and q_len * (h_q / h_kv) <= 16, window >= 0, and the
 * other requirements of paged_gqa_decode; workspace as paged_gqa_decode's.
 * Auto splits: paged_gqa_ext_num_splits (with a window, a grid that fills the
 * GPU is not split; never more shards than paged_gqa_num_splits gives, so its
 * workspace size suffices). */
FP8MLA_API fp8mla_status_t paged_gqa_decode_ext(const void* q, const void* k_cache, const void* v_cache,
                                                fp8mla_kv_dtype_t kv_dtype, int num_blocks, const float* k_scale,
                                                const float* v_scale, int scale_per_row, const int32_t* block_table,
                                                int max_blocks, const int32_t* seqlens, float softmax_scale, int q_len,
                                                const uint8_t* spec_mask, int window, const float* sinks,
                                                int num_splits, void* workspace, size_t workspace_bytes, void* out,
                                                float* lse, int bs, int h_q, int h_kv, int head_dim, int page_size,
                                                fp8mla_stream_t stream);

FP8MLA_API size_t paged_gqa_workspace_bytes(int bs, int h_q, int head_dim, int max_splits);

/* Number of key shards paged_gqa_decode will use for these arguments
 * (num_splits as passed: 0 = auto).  Host-only, no device access. */
FP8MLA_API int paged_gqa_num_splits(int bs, int h_kv, int max_seqlen, int num_sms, int num_splits);

/* Number of key shards paged_gqa_decode_ext will use: paged_gqa_num_splits's
 * rule, except that with a window (window > 0) max_seqlen is taken as the
 * keys the window spans (window + q_len - 1 + 128 at most) and a grid of
 * bs * h_kv CTAs that already fills the GPU is not split (the window makes
 * the sequences' work nearly equal); never more than paged_gqa_num_splits
 * gives for the same arguments.  Host-only. */
FP8MLA_API int paged_gqa_ext_num_splits(int bs, int h_kv, int max_seqlen, int q_len, int window, int num_sms,
                                        int num_splits);

/* ---------------------------------------------------------- cache write ---
 * fp8_paged_cache_write -- quantise-on-write of new K or V rows into an E4M3
 * paged cache (InfiniCore "add FP8 blockwise dequantize/GEMM operators and
 * FP8(E4M3) KV cache support in paged attention", Summary, paged_caching: a
 * write kernel over (token, kv_head) rows; per-row scale amax / 448, 1 when
 * amax is 0, kept in a float32 [num_blocks, h_kv, page] array).
 *   x             bf16 (device): the row of token t, head h starts at element
 *                 t * x_token_stride + h * head_dim and holds head_dim values;
 *                 x 16-byte aligned, x_token_stride a multiple of 8 and
 *                 >= h_kv * head_dim
 *   slot_mapping  int32 [n_tokens] (device): token t goes to block
 *                 slot / page_size, offset slot % page_size.  A negative slot
 *                 skips the token; a slot >= num_blocks * page_size sets
 *                 FP8MLA_DEV_BAD_SLOT and skips it.  Two tokens with the same
 *                 slot race: which one lands is undefined.
 *   cache         E4M3 bytes [num_blocks, h_kv, page_size, head_dim] (device,
 *                 16-byte aligned).  The dense MLA cache [num_pages, 64, 576]
 *                 is h_kv = 1, page_size = 64, head_dim = 576.
 *   exactly one of
 *     tensor_scale  float32 [1] (device): code = E4M3(fp32(x * inv)) with
 *                   inv = fp32(1 / tensor_scale); the value must be a normal
 *                   float > 0 (it is not read on the host)
 *     token_scales  float32 [num_blocks, h_kv, page_size] (device): each
 *                   written row gets scale = fp32(max|x| / 448) (1.0 when the
 *                   row is all zeros), stored at its slot, and
 *                   code = E4M3(fp32(x * inv)) with inv = fp32(448 / max|x|)
 *                   (1.0 for a zero row); a row with max|x| < 2^-64 is first
 *                   multiplied by 2^64 (exact), so inv stays finite
 * Every float operation rounds to nearest even; E4M3 rounding is to nearest
 * even with saturation to +-448.  x must be finite.  head_dim is a multiple
 * of 8 in [8, 1024]; kv_dtype must be FP8MLA_KV_E4M3.  n_tokens = 0 is a
 * no-op.  Bytes and scales of slots no token maps to are not touched.
 * Asynchronous on `stream`; the caller owns every buffer. */
FP8MLA_API fp8mla_status_t fp8_paged_cache_write(const void* x, int64_t x_token_stride, const int32_t* slot_mapping,
                                                 int n_tokens, int h_kv, int head_dim, int page_size,
                                                 int num_blocks, fp8mla_kv_dtype_t kv_dtype, void* cache,
                                                 const float* tensor_scale, float* token_scales,
                                                 fp8mla_stream_t stream);

/* ------------------------------------------------------ no allocation ---
 * fp8mla_decode_no_alloc -- the dense MLA decode for callers that cannot
 * allocate device memory: code running where cudaMalloc is not allowed or
 * not available (inside a host runtime that only hands out fixed input and
 * output buffers, a plugin without access to an allocator, a process with
 * a hard memory budget fixed at start-up).  The pages have no counterpart:
 * this is a deployment convenience of this library.
 *
 * Same arguments and results as fp8mla_decode without the schedule and the
 * workspace: the call schedules one work unit per sequence (no split-KV) and
 * keeps its schedule, split counts and quantised Q in a fixed
 * device array compiled into this library (5.7 MB, held by every GPU that
 * loads the library until the process exits).  It calls no allocator.
 *   b <= FP8MLA_NO_ALLOC_MAX_BATCH; a larger batch returns
 *   FP8MLA_ERR_WORKSPACE_TOO_SMALL and launches nothing.
 *   All calls on a device share the array and it keeps the last call's
 *   contents (every call rewrites what it reads, so nothing needs clearing);
 *   calls that overlap on the GPU (other streams, other host threads) race on
 *   it, so the caller must serialise them.
 *   The first call on each device looks up the array's device address with
 *   that device current (cudaGetSymbolAddress); make that first call before
 *   capturing a stream into a graph. */
#define FP8MLA_NO_ALLOC_MAX_BATCH 64
FP8MLA_API fp8mla_status_t fp8mla_decode_no_alloc(const void* q, const void* kv_cache, fp8mla_kv_dtype_t kv_dtype,
                                                  int num_pages, const int32_t* block_table, int max_pages,
                                                  const int32_t* cache_seqlens, const float* kv_scale,
                                                  float softmax_scale, int causal, void* out, float* lse,
                                                  fp8mla_dot_mode_t dot_mode, int b, int s_q, int h_q,
                                                  fp8mla_stream_t stream);

/* ------------------------------------------------------- measurement ---- */

/* Stage timing of fp8mla_decode, a measurement aid (off by default).  While
 * enabled, fp8mla_decode records CUDA events before and after each of its
 * kernels (Q quantisation, the decode kernel, the combine);
 * those events keep the kernels from overlapping one another, so time the
 * call itself with timing off.  One timer per process, used by one thread at
 * a time: a decode call that times holds it for the call.  Enabling or
 * disabling discards the last record.  Returns FP8MLA_OK. */
FP8MLA_API fp8mla_status_t fp8mla_set_stage_timing(int enable);

/* Synchronises `stream` and writes ms[0..2] = milliseconds of the last timed
 * fp8mla_decode call's Q quantisation, decode kernel and
 * combine.  ms: host pointer to 3 floats.  FP8MLA_ERR_INVALID_ARG if no call
 * was timed since timing was enabled; FP8MLA_ERR_CUDA if the events cannot be
 * read (for instance when the last timed call ran on another device). */
FP8MLA_API fp8mla_status_t fp8mla_get_stage_times(fp8mla_stream_t stream, float* ms);

/* ------------------------------------------------------------- status ---- */

/* Synchronises `stream`, returns in *code_out the OR of the FP8MLA_DEV_* bits
 * recorded since the last call on the current device, and clears them. */
FP8MLA_API fp8mla_status_t fp8mla_get_last_device_error(fp8mla_stream_t stream, uint32_t* code_out);

/* Diagnostics of FP8MLA_DEV_WAIT_TIMEOUT in the dense MLA decode: synchronises
 * `stream` and writes where[0..2] = {source line of the wait, block index,
 * thread index} of the first bounded wait that ran out since the last call
 * on the current device (all 0 if none ran out), then clears the record.
 * where: host pointer to 3 uint32_t. */
FP8MLA_API fp8mla_status_t fp8mla_get_wait_timeout_site(fp8mla_stream_t stream, uint32_t* where);

/* Test hook of the bounded waits (FP8 dot mode of fp8mla_decode and
 * fp8mla_decode_no_alloc), for the current device.  fault_page = p + 1 makes
 * CTA 0 of work unit 0 of every later FP8-dots decode skip the loads of the
 * p-th page of its unit, so the waits on that page run out: the decode then
 * finishes with FP8MLA_DEV_WAIT_TIMEOUT recorded (fp8mla_get_last_device_error)
 * and wrong values in that unit's outputs, and the CUDA context stays usable.
 * fault_page = 0 turns the hook off.  wait_limit_ns sets how long a bounded
 * wait may see no progress before it gives up (0 = the default, 4 s).
 * Not for production use; returns FP8MLA_ERR_CUDA if the symbols cannot be
 * written, FP8MLA_ERR_INVALID_ARG if fault_page < 0. */
FP8MLA_API fp8mla_status_t fp8mla_set_wait_test(int32_t fault_page, uint64_t wait_limit_ns);

/* Static string naming a status code. */
FP8MLA_API const char* fp8mla_status_string(fp8mla_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* FP8MLA_H */
