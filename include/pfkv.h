/*
 * pfkv.h -- C ABI of libpfkv: decode attention over a paged KV cache stored as
 * 8-bit e4m3 floating point and converted back when it is read, for NVIDIA
 * GB300 (sm_103a).
 *
 * Sources of the operations (web pages; section named in each entry below):
 *  - "Inference-engine scheduling explainer": 推論エンジンの実践：Continuous
 *    Batching・Prefix Cache・Speculative Decoding (deepseekmodel.com).
 *  - "Workers AI post": より小さく、高速で、安全に：Kimi と GLM を大規模に展開
 *    するための実行方法 (Cloudflare Workers AI, HN mirror).
 *  - "kLLM article": 快手万擎大模型推理成本和性能优化实践 (6aiq.com).
 *
 * Conventions for every call
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or retains them.  Work is enqueued on `stream`
 *    (asynchronous; no call synchronises unless its comment says so).
 *  - bf16 = IEEE bfloat16 bit patterns (uint16); e4m3 = OCP 8-bit E4M3 codes
 *    (uint8: bias 7, subnormals, 0x7F/0xFF NaN, no infinity, max 448).
 *  - Layouts are row-major (C order) with the shapes written in brackets.
 *  - Alignment: bf16 and e4m3 tensors start on 16 bytes, workspaces on 256,
 *    int32 / uint32 / fp32 arrays on 4 and int64 slot mappings on 8 (device
 *    scale arrays as their call says); a pointer that is not is rejected with
 *    PFKV_ERR_INVALID_ARG before anything is enqueued.
 *  - Paged caches: K and V are separate tensors [num_pages][Hkv][P][D]; the
 *    token at logical position t of request b lives in page
 *    block_tables[b][t / P], row t % P ("slot" = page * P + t % P).  The MLA
 *    latent cache is [num_pages][P][Dqk] (the same layout with Hkv = 1).
 *    A cache holds at least one page: num_pages < 1 is rejected with
 *    PFKV_ERR_INVALID_ARG, also by a call that would have nothing to do.
 *  - context_lens[b] counts every token attended, including tokens appended
 *    in the same step.
 *  - Return value: PFKV_OK, or a negative pfkv_status for argument, support or
 *    launch errors, detected synchronously before anything is enqueued (a
 *    launch error after enqueueing is reported as PFKV_ERR_CUDA).
 *    pfkv_last_error() gives a message for the calling thread.
 *  - Data errors that only the GPU can see (a block-table entry outside the
 *    pool, a top-k index beyond the context) never cause an out-of-bounds
 *    access: the kernels clamp or skip, and set a bit in the status word at the
 *    start of the workspace (read it with pfkv_workspace_status) or, for
 *    pfkv_validate_tables, in the caller's error word.
 *  - No kernel spins on memory written by another kernel.  Intra-kernel
 *    barrier waits are bounded (about one second); on expiry the kernel sets
 *    PFKV_DEVERR_WAIT_TIMEOUT and returns.
 */
#ifndef PFKV_H
#define PFKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PFKV_API __attribute__((visibility("default")))
#else
#define PFKV_API
#endif

/* CUDA stream handle (cudaStream_t); declared opaquely so that this header
 * does not require the CUDA headers.  NULL is the legacy default stream. */
typedef struct CUstream_st *pfkv_stream_t;

typedef enum {
  PFKV_OK = 0,
  PFKV_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad shape */
  PFKV_ERR_UNSUPPORTED = -2, /* valid but not implemented (head_dim, page size, ...) */
  PFKV_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed */
  PFKV_ERR_INDEX = -4,       /* an index error was found (status word set) */
  PFKV_ERR_WORKSPACE = -5,   /* workspace too small for this call */
  PFKV_ERR_NO_PAGES = -6     /* the page pool has too few free pages */
} pfkv_status;

typedef enum { PFKV_CACHE_FP8_E4M3 = 0, PFKV_CACHE_BF16 = 1 } pfkv_cache_dtype;

/* Bits of the device status word (workspace header / validation word). */
#define PFKV_DEVERR_WAIT_TIMEOUT 0x01 /* a bounded barrier wait expired */
#define PFKV_DEVERR_BAD_PAGE 0x02     /* block-table entry outside [0, num_pages) */
#define PFKV_DEVERR_BAD_CONTEXT 0x04  /* context_lens[b] < 0 or > max_pages_per_seq * P */
#define PFKV_DEVERR_WORKSPACE 0x08    /* partial-state slots exceeded the workspace */
#define PFKV_DEVERR_BAD_TOPK 0x10     /* top-k index >= context length */
#define PFKV_DEVERR_BAD_SLOT 0x20     /* slot_mapping entry >= num_pages * P */

/* ------------------------------------------------------------------------ */
/* kv_append_fp8 -- quantise new K/V rows to e4m3 and scatter them into pages.
 *
 * Workers AI post, §1 "KV キャッシュの量子化": the cache holds 8-bit e4m3
 * instead of BF16, halving its size.  Inference-engine scheduling explainer,
 * section "FP8 KV のエンジニアリング上の制約": the scale is per tensor, per head
 * or per token; this call takes one fp32 scale per tensor (one for K, one for
 * V).  Section "PagedAttention の 2 つの原語": KV goes to fixed-size pages
 * through a slot mapping.
 *
 * For token i < num_tokens, head h, element d:
 *     code = e4m3_rne_satfinite( fp32(x[i][h][d]) / scale )   (IEEE fp32 divide)
 * stored at cache[slot / P][h][slot % P][d] with slot = slot_mapping[i].
 *   k_new, v_new   bf16 [num_tokens][num_kv_heads][head_dim]
 *   k_cache, v_cache  e4m3 [num_pages][num_kv_heads][page_size][head_dim]
 *   slot_mapping   int64 [num_tokens]; slot < 0 skips the token; a slot
 *                  >= num_pages * page_size is skipped (nothing is written).
 * One latent tensor (MLA cKV): pass v_new = v_cache = NULL, num_kv_heads = 1,
 * head_dim = Dqk; v_scale is then ignored.
 * Supported: head_dim a multiple of 16, page_size >= 1, scales > 0 and finite.
 * Errors: PFKV_ERR_INVALID_ARG for null k pointers, num_tokens < 0, bad dims
 * or scales.  num_tokens == 0 enqueues nothing. */
PFKV_API int pfkv_kv_append_fp8(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                       const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                       int head_dim, int page_size, int64_t num_pages, float k_scale,
                       float v_scale, pfkv_stream_t stream);

/* Same scatter into a bf16 cache (no quantisation), for the BF16-cache
 * comparison the Workers AI post makes (§1: FP8 halves the cache bytes). */
PFKV_API int pfkv_kv_append_bf16(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                        const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                        int head_dim, int page_size, int64_t num_pages, pfkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Scale granularity of an e4m3 cache.
 *
 * Explainer, section "FP8 KV のエンジニアリング上の制約": the scaling factor can
 * be per tensor, per head or per token; the finer it is, the more precise the
 * cache and the more extra work and memory traffic inside the decode kernel.
 * The section lists the three from coarse to fine, so per token is read as
 * finer than per head: one scale for every (token, KV head) row.  Scales are
 * fp32 DEVICE arrays:
 *   PFKV_SCALE_TENSOR  [1]
 *   PFKV_SCALE_HEAD    [num_kv_heads]
 *   PFKV_SCALE_TOKEN   [num_pages][num_kv_heads][page_size], entry
 *                      (page * num_kv_heads + h) * page_size + offset beside
 *                      the cache row it scales */
typedef enum {
  PFKV_SCALE_TENSOR = 0,
  PFKV_SCALE_HEAD = 1,
  PFKV_SCALE_TOKEN = 2
} pfkv_scale_granularity;

/* kv_append_fp8_scaled -- kv_append_fp8 with device-resident scales.
 *  TENSOR, HEAD: k_scales / v_scales are READ (scale = scales[0] or
 *      scales[h]); code = e4m3_rne_satfinite(fp32(x) / scale).  Scales must be
 *      finite and > 0 (not checked: they live on the device).
 *  TOKEN: k_scales / v_scales are WRITTEN, one entry per appended row:
 *      s = fp32(max_d |x[i][h][d]|) / 448 (IEEE fp32 divide), then
 *      code = e4m3_rne_satfinite(fp32(x) / s), so the row's largest magnitude
 *      becomes the largest e4m3 value; an all-zero row stores s = 0 and zero
 *      codes.  Inputs must be finite.
 * Other arguments, layouts and skipped slots as kv_append_fp8; v_new = v_cache
 * = v_scales = NULL appends K only.
 * Supported: head_dim a multiple of 16 (TOKEN: at most 512); scale arrays
 * 4-byte aligned.  Errors: PFKV_ERR_INVALID_ARG for an unknown granularity or
 * a NULL scale array, plus those of kv_append_fp8. */
PFKV_API int pfkv_kv_append_fp8_scaled(const void *k_new, const void *v_new, void *k_cache,
                                       void *v_cache, const int64_t *slot_mapping, int num_tokens,
                                       int num_kv_heads, int head_dim, int page_size,
                                       int64_t num_pages, pfkv_scale_granularity granularity,
                                       float *k_scales, float *v_scales, pfkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* paged_decode_attn -- one decode step of GQA/MHA attention over the paged
 * cache, dequantising on read, with split-KV and a log-sum-exp merge.
 *
 * Explainer, "PagedAttention の 2 つの原語": the kernel resolves KV addresses
 * through block_table.  Workers AI post, §1: the FP8 attention kernel converts
 * values as it reads them.  kLLM article, §5.2.2: blockwise attention keeps
 * (m, ℓ, O) per block so that the merged result equals full attention.
 *
 * For request b, query head h (KV head kvh = h / (Hq / Hkv)), t < L_b:
 *   s_t  = softmax_scale * sum_d q[b][h][d] * K(t)[d] * k_scale
 *   out  = sum_t e^{s_t - m} V(t) * v_scale / sum_t e^{s_t - m}
 *   lse  = m + ln sum_t e^{s_t - m}          (m = max_t s_t; natural log)
 * where K(t)/V(t) are the e4m3 (or bf16) rows at block_tables[b][t / P].
 * The work is split into contiguous runs of 16-token tiles balanced over all
 * warps of a persistent grid; runs that do not cover a whole request write
 * fp32 partial states to the workspace and a merge kernel combines them.
 *   out            bf16 [batch][num_q_heads][head_dim]
 *   q              bf16 [batch][num_q_heads][head_dim]
 *   k_cache/v_cache  e4m3 or bf16 [num_pages][num_kv_heads][page_size][head_dim]
 *   block_tables   int32 [batch][max_pages_per_seq]
 *   context_lens   int32 [batch] (device)
 *   kv_split_tokens  0: split only for balance; > 0: additionally cut every
 *                  request into chunks of this many tokens, each merged by
 *                  log-sum-exp (must be a multiple of 16)
 *   lse_out        optional fp32 [batch][num_q_heads] (NULL: not written)
 *   workspace      device scratch of at least pfkv_paged_decode_workspace_size()
 *                  bytes, 256-byte aligned; contents on entry are ignored.
 * L_b == 0 gives out = 0 and lse = -inf.  For a bf16 cache the scales still
 * multiply (pass 1.0).
 * Numerics: fp32 accumulation throughout.  e4m3 cache: scores are e4m3
 * products on the cached K bytes against q split into two e4m3 parts after a
 * power-of-two scale per query head (largest |q| into (224, 448]; exact for
 * every value at least 1/896 of the head's largest, within 2^-10 of the scaled
 * value below that; any finite bf16 q is accepted, 1 / scale multiplies the raw
 * scores); P.V takes f16 products (V widens exactly, P <= 2^8).  bf16 cache:
 * bf16 products for both.
 * Supported: head_dim 128; page_size a multiple of 16; num_q_heads /
 * num_kv_heads in 1..16; num_pages * num_kv_heads * page_size < 2^31.
 * Device errors (status word): PFKV_DEVERR_BAD_PAGE (rows outside the pool
 * read as zeros), PFKV_DEVERR_BAD_CONTEXT (length clamped to the table),
 * PFKV_DEVERR_WORKSPACE, PFKV_DEVERR_WAIT_TIMEOUT. */
PFKV_API size_t pfkv_paged_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads,
                                        int head_dim, int kv_split_tokens,
                                        int64_t max_total_chunks);
PFKV_API int pfkv_paged_decode_attn(void *out, const void *q, const void *k_cache, const void *v_cache,
                           pfkv_cache_dtype cache_dtype, const int32_t *block_tables,
                           int max_pages_per_seq, const int32_t *context_lens, int batch,
                           int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                           int64_t num_pages, float k_scale, float v_scale, float softmax_scale,
                           int kv_split_tokens, void *workspace, size_t workspace_bytes,
                           float *lse_out, pfkv_stream_t stream);

/* paged_decode_attn_noalloc -- the same computation as pfkv_paged_decode_attn
 * for callers that cannot allocate device memory where decode runs (an engine
 * that reserves all device memory up front and hands out every byte from its
 * own pool, or a per-token path that cannot afford the synchronisation and
 * latency of cudaMalloc).  The source pages have no counterpart of this call;
 * it exists for such callers only.
 *  - Scratch is a fixed 64 MiB array inside the library's device module,
 *    present on every GPU that loads the library until the process exits.
 *    A call whose pfkv_paged_decode_workspace_size(batch, num_q_heads,
 *    num_kv_heads, head_dim, kv_split_tokens, max_total_chunks) exceeds 64 MiB
 *    fails with PFKV_ERR_WORKSPACE and enqueues nothing.
 *  - The call allocates nothing (no cudaMalloc, no allocating library call).
 *    Its first call on a device looks up the array's device address on that
 *    device (cudaGetSymbolAddress); make that first call before any stream
 *    capture begins.
 *  - All calls share the one array.  Two calls whose work overlaps on the GPU
 *    (different streams without ordering between them) race on it; order them.
 *  - status_out: optional device int32 that receives the device status word
 *    (PFKV_DEVERR_* bits) of this call, copied after the decode on `stream`;
 *    for batch == 0 it is set to 0 on `stream`.
 *  - The array's device address is looked up once per device and kept for
 *    the life of the process: resetting a device (cudaDeviceReset) while the
 *    library is loaded is not supported, since later calls would use the
 *    address the reset invalidated.
 *  - Other arguments, layouts and errors as pfkv_paged_decode_attn. */
PFKV_API int pfkv_paged_decode_attn_noalloc(void *out, const void *q, const void *k_cache,
                                            const void *v_cache, pfkv_cache_dtype cache_dtype,
                                            const int32_t *block_tables, int max_pages_per_seq,
                                            const int32_t *context_lens, int batch, int num_q_heads,
                                            int num_kv_heads, int head_dim, int page_size,
                                            int64_t num_pages, float k_scale, float v_scale,
                                            float softmax_scale, int kv_split_tokens,
                                            int64_t max_total_chunks, float *lse_out,
                                            int32_t *status_out, pfkv_stream_t stream);

/* paged_decode_attn_scaled -- paged_decode_attn over an e4m3 cache whose
 * scales are device arrays of the given granularity (see
 * pfkv_scale_granularity):
 *   s_t = softmax_scale * sum_d q[b][h][d] * e4m3(Kcode_t[d]) * ks(t)
 *   out = sum_t e^{s_t - m} e4m3(Vcode_t[d]) * vs(t) / sum_t e^{s_t - m}
 * with ks(t), vs(t) = scales[0], scales[kvh] or the scale stored beside row t.
 * Per tensor and per head, the scales fold into the score and output factors
 * of each work unit, so the tile loop is unchanged.  Per token, the 16 K and
 * 16 V scales of each 16-token tile (2 x 64 bytes) are copied in with the
 * tile: 8 extra bytes per (token, KV head) against 2 x head_dim bytes of
 * codes; each K scale multiplies its raw score, and each V scale, relative to
 * the largest V scale seen so far in the work unit, multiplies its token's
 * probability before the f16 P.V product (the accumulator is rescaled when
 * that largest scale grows, as for the running maximum of the softmax).
 * Numerics: per tensor and per head as pfkv_paged_decode_attn; per token, the
 * score products are f16 on K widened in registers, against q times one
 * power of two per work unit that takes its largest |q| into (2^14, 2^15]
 * (any finite bf16 q; exact for every value at least 2^-29 of that largest).
 * Scales: finite and >= 0 (TENSOR, HEAD: > 0); not checked (device arrays).
 * The scale of a token past L_b is never used.  Workspace: as
 * pfkv_paged_decode_attn (pfkv_paged_decode_workspace_size).  Other arguments
 * and device errors as pfkv_paged_decode_attn; a row outside the pool reads as
 * zeros with zero scales.
 * Supported: as pfkv_paged_decode_attn, e4m3 cache only; scale arrays 16-byte
 * aligned. */
PFKV_API int pfkv_paged_decode_attn_scaled(void *out, const void *q, const void *k_cache,
                                           const void *v_cache,
                                           pfkv_scale_granularity granularity,
                                           const float *k_scales, const float *v_scales,
                                           const int32_t *block_tables, int max_pages_per_seq,
                                           const int32_t *context_lens, int batch,
                                           int num_q_heads, int num_kv_heads, int head_dim,
                                           int page_size, int64_t num_pages, float softmax_scale,
                                           int kv_split_tokens, void *workspace,
                                           size_t workspace_bytes, float *lse_out,
                                           pfkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* paged_prefill_attn -- several new query tokens per request over the paged
 * e4m3 cache, causal among the new tokens: the attention of a chunked-prefill
 * step or of a speculative-decoding verification pass.
 *
 * Explainer, section "チャンク分割と、その大きさの決め方": a chunked prefill
 * writes each chunk's KV before the next, and the chunk's tokens attend the
 * cached prefix and each other; "Speculative Decoding" section: the target
 * model checks the gamma+1 drafted positions in one parallel forward pass.
 * kLLM article, §5.2.2: chunks of a long context merge by (m, ℓ, O).
 *
 * Request b has n_b = q_start[b+1] - q_start[b] query tokens, at positions
 * L_b - n_b .. L_b - 1 (their K/V must already be in the cache: append them
 * first).  For query i of request b and query head h (kvh = h / (Hq / Hkv)):
 *   s_t = softmax_scale * sum_d q[q_start[b]+i][h][d] * K(t)[d] * k_scale,
 *         t = 0 .. L_b - n_b + i
 *   out = sum_t e^{s_t - m} V(t) * v_scale / sum_t e^{s_t - m}
 *   lse = m + ln sum_t e^{s_t - m}
 * Products on the tensor cores with fp32 accumulation.  Scores: e4m3
 * products on the K bytes with each q row, scaled by a power of two (largest
 * |q| into (224, 448]), split into two e4m3 parts (exact for every value at
 * least 1/896 of the row's largest, within 2^-10 of the scaled value below
 * that); any finite bf16 q is accepted and 1 / scale multiplies the raw
 * scores.  P.V: f16 (P <= 2^8, V widened exactly).
 *   out, q        bf16 [q_start[batch]][num_q_heads][head_dim]
 *   q_start       int32 [batch + 1] (device), non-decreasing, q_start[0] = 0
 *   max_q_len     host bound on every n_b; max_context_len host bound on
 *                 every L_b (the grid is sized from them; larger values are
 *                 clamped and flagged PFKV_DEVERR_BAD_CONTEXT, as is n_b > L_b)
 *   kv_split_tokens  0: one pass over each request's context; > 0 (a
 *                 multiple of 64): chunks of that many tokens run in parallel
 *                 and are merged (workspace grows with batch * num_kv_heads *
 *                 ceil(max_q_len * G / 128) * ceil(max_context_len / split)).
 *                 Not used when max_q_len * G <= 64 (verification-sized
 *                 calls): the contexts of all (request, KV head) pairs are
 *                 then split evenly over one CTA per SM and the pieces merged
 *                 (workspace: (SMs of the current device + batch *
 *                 num_kv_heads) 64-row partial states plus batch + 1
 *                 offsets, so query the size on the device that will run the
 *                 call), whatever the value (it is still checked)
 *   workspace     >= pfkv_paged_prefill_workspace_size(...) bytes, 256-byte
 *                 aligned; lse_out optional fp32 [q_start[batch]][num_q_heads]
 * Other layouts as pfkv_paged_decode_attn.
 * Supported: head_dim 128; e4m3 cache; page_size a multiple of 16;
 * (num_q_heads / num_kv_heads) divides 128.
 * Device errors: PFKV_DEVERR_BAD_PAGE (rows read as zeros),
 * PFKV_DEVERR_BAD_CONTEXT, PFKV_DEVERR_WAIT_TIMEOUT. */
PFKV_API size_t pfkv_paged_prefill_workspace_size(int batch, int num_q_heads, int num_kv_heads,
                                                  int head_dim, int max_q_len, int max_context_len,
                                                  int kv_split_tokens);
PFKV_API int pfkv_paged_prefill_attn(void *out, const void *q, const void *k_cache,
                                     const void *v_cache, const int32_t *block_tables,
                                     int max_pages_per_seq, const int32_t *context_lens,
                                     const int32_t *q_start, int batch, int num_q_heads,
                                     int num_kv_heads, int head_dim, int page_size,
                                     int64_t num_pages, int max_q_len, int max_context_len,
                                     float k_scale, float v_scale, float softmax_scale,
                                     int kv_split_tokens, void *workspace, size_t workspace_bytes,
                                     float *lse_out, pfkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* mla_decode_attn -- MLA absorbed-latent decode over one shared e4m3 latent
 * row per token, optionally restricted to a top-k token list.
 *
 * kLLM article, §5.1.1: DSA selects the top-k historical tokens that take part
 * in attention and MLA keeps a compressed per-token cKV; §5.1.2: that cKV is
 * shared by all heads.  Absorbed reading: the whole Dqk-wide row is the key,
 * its first d_latent entries are the value.
 *   s_t = softmax_scale * sum_{d<Dqk} q[b][h][d] * c_t[d] * ckv_scale
 *   out = sum_t e^{s_t - m} c_t[0:d_latent] * ckv_scale / sum_t e^{s_t - m}
 * over t in topk_idx[b][0:topk] (entries < 0 are padding and skipped), or over
 * every t < L_b when topk_idx is NULL.  Dqk = d_latent + d_rope.
 *   out        bf16 [batch][num_heads][d_latent]
 *   q          bf16 [batch][num_heads][Dqk]
 *   ckv_cache  e4m3 [num_pages][page_size][Dqk]
 *   topk_idx   int32 [batch][topk] or NULL
 *   lse_out    optional fp32 [batch][num_heads]
 * Supported: d_latent 512, d_rope 64, num_heads 128 or fewer and a multiple of
 * 16, page_size a multiple of 16, num_pages * page_size < 2^31.  Listed
 * indices >= L_b are skipped and set PFKV_DEVERR_BAD_TOPK.
 * Numerics: f16 operands with f32 accumulation: the latent widens exactly; a q
 * row converts as it is when its largest |q| over the columns one SM contracts
 * lies in [2^-4, 2^15] (then every value at least 2^-10 of that largest is
 * exact), otherwise after a power-of-two scale into (2^14, 2^15] that the
 * SM's partial scores undo; any finite bf16 q is accepted.  Each request runs on a pair
 * of SMs that each contract part of the 576 columns; a score is one SM's
 * exact f32 partial plus the other's partial carried as 16-bit fixed point
 * over its range within a 32-token tile (at most range / 65535 added error,
 * in log2 units).
 * Small batches: when 2 * batch SMs leave pairs of SMs idle, each request's
 * list is split into runs of at least 256 positions handled by separate
 * pairs, whose (reference, sum, unnormalised output) states are folded by
 * log-sum-exp in a second kernel (kLLM article §5.2.2: blockwise states
 * combine to full attention).  pfkv_mla_decode_workspace_size returns the
 * status word plus room for those states (batch * splits * num_heads * 2064
 * bytes, splits chosen from the current device's SM count); with a smaller
 * workspace (at least 256 bytes) the call uses as many splits as fit, down
 * to one.  The split changes only the order of the softmax sums. */
PFKV_API size_t pfkv_mla_decode_workspace_size(int batch, int num_heads, int d_latent, int topk);
PFKV_API int pfkv_mla_decode_attn(void *out, const void *q, const void *ckv_cache,
                         const int32_t *block_tables, int max_pages_per_seq,
                         const int32_t *context_lens, const int32_t *topk_idx, int topk,
                         int batch, int num_heads, int d_latent, int d_rope, int page_size,
                         int64_t num_pages, float ckv_scale, float softmax_scale,
                         void *workspace, size_t workspace_bytes, float *lse_out,
                         pfkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* validate_tables -- opt-in index check before decode (Workers AI post, §3
 * "共用 KV キャッシュの保護": verify the request-to-page mapping before reading,
 * as a separate batched check rather than inside the attention kernel).
 * Zeroes *d_err_word, then ORs PFKV_DEVERR_* bits for: context_lens out of
 * range, a block-table entry used by some request outside [0, num_pages), a
 * top-k index >= its context length (topk_idx may be NULL), a slot_mapping
 * entry >= num_pages * page_size (slot_mapping may be NULL).  d_err_word is a
 * device int32; read it after the stream reaches this point. */
PFKV_API int pfkv_validate_tables(const int32_t *block_tables, int max_pages_per_seq,
                         const int32_t *context_lens, int batch, int page_size, int64_t num_pages,
                         const int32_t *topk_idx, int topk, const int64_t *slot_mapping,
                         int num_slots, int32_t *d_err_word, pfkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* verify_page_tags -- KV page integrity check before decode (Workers AI post,
 * §3 "共用 KV キャッシュの保護", 動作原理): every physical page carries a tag
 * that changes each time the page is handed out again; right before decode
 * reads the cache, each request's pages are checked against the tags the
 * request recorded when it mapped them, and a request that fails is aborted
 * instead of reading another request's data.  A separate batched kernel, not
 * fused into attention (the post's cost argument).
 *   block_tables    int32  [batch][max_pages_per_seq]  device
 *   table_tags      uint32 [batch][max_pages_per_seq]  device: tag recorded with each entry
 *   context_lens    int32  [batch]                     device
 *   page_tags       uint32 [num_pages]                 device: current tag of each page
 *   request_status  int32  [batch]                     device, written: 0 (ok) or an OR of
 *     PFKV_REQ_TAG_MISMATCH  a page the request reads (entry i < ceil(L / page_size)) carries
 *                            a different tag now
 *     PFKV_REQ_BAD_INDEX     such an entry is outside [0, num_pages), or L < 0 or
 *                            L > max_pages_per_seq * page_size
 * Entries past a request's context are not read and not checked.  Asynchronous
 * on `stream`; the caller reads request_status after the stream reaches this
 * point and leaves flagged requests out of the decode call.  Returns PFKV_OK,
 * PFKV_ERR_INVALID_ARG (bad sizes, a NULL or not 4-byte aligned pointer) or
 * PFKV_ERR_CUDA. */
#define PFKV_REQ_TAG_MISMATCH 0x1
#define PFKV_REQ_BAD_INDEX 0x2
PFKV_API int pfkv_verify_page_tags(const int32_t *block_tables, const uint32_t *table_tags,
                                   int max_pages_per_seq, const int32_t *context_lens, int batch,
                                   int page_size, const uint32_t *page_tags, int64_t num_pages,
                                   int32_t *request_status, pfkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Page pool and prefix cache (host side; no device memory, no CUDA calls).
 * KV cache explainer, "PagedAttention の 2 つの原語": the cache is a pool of
 * fixed-size pages plus per-request block tables; allocating is popping a page
 * id off a free list and freeing is pushing it back (O(1), no device
 * allocation); pages can be shared.  "Prefix Cache" section: each full block
 * is identified by a hash of its tokens chained through its parent block's
 * hash, a lookup walks a prompt's blocks in order and stops at the first miss,
 * so the reused length is floored to whole blocks (100 shared tokens with
 * 16-token blocks reuse 96).
 * The pool keeps a reference count per page (a shared page returns to the free
 * list when its last holder releases it, and then leaves the prefix table) and
 * a generation tag per page that changes each time the page is handed out:
 * the tags pfkv_verify_page_tags checks.  Not thread-safe.
 * Block hash: 64-bit FNV-1a over the parent hash (8 bytes little endian) then
 * the block's token ids (4 bytes each, little endian); the first block's
 * parent is 0. */
typedef struct pfkv_page_pool pfkv_page_pool;
/* A pool of num_pages pages of page_size tokens, all free; NULL on bad sizes
 * (message in pfkv_last_error).  Free pages are handed out lowest id first. */
PFKV_API pfkv_page_pool *pfkv_pool_create(int64_t num_pages, int page_size);
PFKV_API void pfkv_pool_destroy(pfkv_page_pool *pool);
/* Free pages left (-1 for a NULL pool). */
PFKV_API int64_t pfkv_pool_num_free(const pfkv_page_pool *pool);
/* Holders of `page` (-1 if out of range). */
PFKV_API int pfkv_pool_refcount(const pfkv_page_pool *pool, int32_t page);
/* Current generation tag of every page into tags_out[num_pages] (host). */
PFKV_API int pfkv_pool_page_tags(const pfkv_page_pool *pool, uint32_t *tags_out);
/* Map a request's token stream (host int32 [n_tokens]) onto pages: the
 * longest run of leading full blocks found in the prefix table is shared (each
 * such page gains a holder), every other block gets a fresh page, and fresh
 * full blocks enter the prefix table.  Writes block_table_row[max_pages]
 * (page ids, -1 past the last page) and table_tags[max_pages] (the tag of each
 * mapped page, 0 past it), and *cached_tokens = shared blocks x page_size.
 * PFKV_ERR_NO_PAGES (nothing changed) if the free list is too short;
 * PFKV_ERR_INVALID_ARG if the row is too short. */
PFKV_API int pfkv_pool_map_request(pfkv_page_pool *pool, const int32_t *tokens, int n_tokens,
                                   int32_t *block_table_row, uint32_t *table_tags, int max_pages,
                                   int *cached_tokens);
/* Release a request's first n_pages pages (one holder per entry: a page
 * listed k times drops k holders); pages with no holder left return to the
 * free list.  PFKV_ERR_INVALID_ARG (nothing changed) if an entry is not a held
 * page, or lists a page more times than it has holders. */
PFKV_API int pfkv_pool_release(pfkv_page_pool *pool, const int32_t *block_table_row, int n_pages);
/* The FNV-1a chain hash of one block (n tokens) given its parent's hash. */
PFKV_API uint64_t pfkv_block_hash(uint64_t parent, const int32_t *tokens, int n);
/* slots_out[k] = page * page_size + t % page_size for tokens t = first_token +
 * k of a request (host arrays): the slot mapping kv_append_fp8 takes. */
PFKV_API int pfkv_slots_from_table(const int32_t *block_table_row, int max_pages, int page_size,
                                   int first_token, int n_tokens, int64_t *slots_out);

/* Copy the workspace status word (bits PFKV_DEVERR_*) to *status after
 * synchronising `stream`.  Returns PFKV_OK, or PFKV_ERR_CUDA. */
PFKV_API int pfkv_workspace_status(const void *workspace, int32_t *status, pfkv_stream_t stream);

/* Diagnostic: one thread waits, with the bounded wait every kernel uses, on a
 * barrier that nothing completes; after about one second it gives up and
 * writes PFKV_DEVERR_WAIT_TIMEOUT to *d_status (device int32).  Shows that an
 * expired wait ends the kernel with a status instead of hanging the GPU.  The
 * pages have no counterpart of this call. */
PFKV_API int pfkv_selftest_barrier_timeout(int32_t *d_status, pfkv_stream_t stream);

/* Message describing the last error on the calling thread ("" if none). */
PFKV_API const char *pfkv_last_error(void);

/* Library version string. */
PFKV_API const char *pfkv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PFKV_H */
