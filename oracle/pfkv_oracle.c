/*
 * pfkv_oracle.c -- plain, slow, obviously-correct CPU oracle for paged FP8 (e4m3)
 * KV decode attention.  TEST INFRASTRUCTURE ONLY: only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this library.  The product
 * path (libpfkv) neither links nor calls it, and shares no code with it.
 *
 * Everything here is written from the definitions on the source pages:
 *
 *  [KVB]  Inference-engine scheduling explainer, "推論エンジンの実践：Continuous
 *         Batching・Prefix Cache・Speculative Decoding", section
 *         "算力利用率が低いのは表の現象、メモリウォールが根因" (KV bytes ≈
 *         2 × layers × KV heads × head_dim × seq × bytes per element).
 *  [PAGE] same page, section "PagedAttention の 2 つの原語": fixed-size blocks
 *         (16 tokens by default), a block_table mapping logical block -> physical
 *         block, and the attention kernel resolving KV addresses through it.
 *  [FP8]  Workers AI post "より小さく、高速で、安全に：Kimi と GLM を大規模に展開
 *         するための実行方法", §1 "KV キャッシュの量子化": the cache is stored as
 *         8-bit floating point in the e4m3 format and the attention kernel
 *         converts values when it reads them.
 *  [SCL]  explainer page, section "FP8 KV のエンジニアリング上の制約": scaling
 *         factors per tensor, per head or per token (all three here).
 *  [OSM]  Kuaishou kLLM article "快手万擎大模型推理成本和性能优化实践", §5.2.2
 *         "分块式 Ring Attention 实现": blockwise attention keeps the running
 *         maximum, normaliser and output (m, ℓ, O) so that the blockwise result
 *         equals full attention.
 *  [CHK]  explainer page, section "チャンク分割と、その大きさの決め方": chunked
 *         prefill cuts a prompt into fixed-size chunks, one per step, writing
 *         each chunk's KV before the next; its tokens attend the cached prefix
 *         and each other causally.
 *  [SPEC] same page, "Speculative Decoding" section: the target model checks
 *         the gamma+1 drafted positions in one parallel forward pass.
 *  [MLA]  same article, §5.1.1/§5.1.2: MLA keeps one compressed latent cKV per
 *         token shared by all heads; DSA selects the top-k historical tokens that
 *         take part in attention.
 *
 * Precision: all attention arithmetic is IEEE double.  The quantiser follows the
 * fp32 path that the append step defines (bf16 -> fp32, fp32 division by the
 * per-tensor scale, one rounding to e4m3), because the stored byte is the
 * product of that fp32 computation; the rounding itself is done by exact
 * comparison against the decoded grid in double.
 *
 * Build: gcc -std=c11 -O1 -ffp-contract=off -fno-fast-math -shared -fPIC
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "pfkv_oracle.h"

/* ------------------------------------------------------------------------- */
/* e4m3 format ([FP8]).  The pages name the format only ("e4m3"); the reading
 * taken is the OCP 8-bit E4M3 format that GPUs implement: 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal
 * (value = m / 8 * 2^-6); the pattern S.1111.111 is NaN; there are no
 * infinities, so the largest finite magnitude is 1.75 * 2^8 = 448 (0x7E).      */

double orc_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);           /* subnormal */
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);  /* normal */
    return sign ? -mag : mag;
}

/* Round an fp32 value to the nearest e4m3 value, ties to the even mantissa,
 * saturating to +-448 instead of overflowing (the format has no infinity);
 * NaN maps to 0x7F.  Found by exact comparison with the decoded grid. */
uint8_t orc_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    /* magnitudes of codes 0x00..0x7E increase strictly with the code: find the
     * largest code lo with value(lo) <= a by bisection over the grid */
    int lo = 0, hi = 0x7E; /* value(lo) <= a < value(hi) (a < 448 here) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (orc_e4m3_value((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    /* value(lo) <= a < value(lo+1) */
    double vlo = orc_e4m3_value((uint8_t)lo);
    double vhi = orc_e4m3_value((uint8_t)(lo + 1));
    int pick;
    if (a - vlo < vhi - a)
        pick = lo;
    else if (a - vlo > vhi - a)
        pick = lo + 1;
    else
        pick = (lo % 2 == 0) ? lo : lo + 1; /* tie: even mantissa (code LSB) */
    return (uint8_t)(sign | pick);
}

/* The same rounding applied to each element of an array. */
void orc_e4m3_encode_array(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_e4m3_encode(x[i]);
}

float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------- */
/* Append ([FP8], [SCL], [PAGE]): quantise each new element as
 *   code = e4m3(fp32(x) / scale)
 * and store it at slot = physical_page * P + offset in the cache laid out as
 * [num_pages][H][P][D].  A negative slot means "skip this token". */
int orc_kv_append(const uint16_t *x_new, uint8_t *cache, const int64_t *slot_mapping,
                  int T, int H, int D, int P, int64_t num_pages, float scale)
{
    for (int t = 0; t < T; t++) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_pages * (int64_t)P)
            return ORC_ERR_INDEX;
        int64_t page = slot / P;
        int64_t off = slot % P;
        for (int h = 0; h < H; h++) {
            for (int d = 0; d < D; d++) {
                float x = orc_bf16_to_f32(x_new[((int64_t)t * H + h) * D + d]);
                float y = x / scale; /* IEEE single-precision division */
                cache[((page * H + h) * P + off) * D + d] = orc_e4m3_encode(y);
            }
        }
    }
    return ORC_OK;
}

/* Same append for a bf16 cache: the element is stored unchanged. */
int orc_kv_append_bf16(const uint16_t *x_new, uint16_t *cache, const int64_t *slot_mapping,
                       int T, int H, int D, int P, int64_t num_pages)
{
    for (int t = 0; t < T; t++) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_pages * (int64_t)P)
            return ORC_ERR_INDEX;
        int64_t page = slot / P;
        int64_t off = slot % P;
        for (int h = 0; h < H; h++)
            for (int d = 0; d < D; d++)
                cache[((page * H + h) * P + off) * D + d] = x_new[((int64_t)t * H + h) * D + d];
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Finer scale granularities ([SCL]): one scale per tensor, one per KV head, or
 * one per token.  The section lists the three in order of increasing fineness,
 * so "per token" is read as finer than "per head": one scale for each
 * (token, KV head) row of D values.  Where the scales live:
 *   ORC_SCALE_TENSOR  scales[0]
 *   ORC_SCALE_HEAD    scales[h]                               h = KV head
 *   ORC_SCALE_TOKEN   scales[(page * H + h) * P + off]   beside the cache row
 * The per-token scale maps the row's largest magnitude onto the largest e4m3
 * value, s = fp32(max_d |x_d|) / 448 (fp32 division), the same amax / 448 rule
 * the per-tensor scale follows over a whole tensor; an all-zero row gets s = 0
 * and zero codes (nothing to scale). */
static double scale_at(int granularity, const float *scales, int64_t cache_row, int h)
{
    if (granularity == ORC_SCALE_TENSOR)
        return (double)scales[0];
    if (granularity == ORC_SCALE_HEAD)
        return (double)scales[h];
    return (double)scales[cache_row];
}

/* Append with one given scale per KV head: code = e4m3(fp32(x) / scales[h]). */
int orc_kv_append_head(const uint16_t *x_new, uint8_t *cache, const float *head_scales,
                       const int64_t *slot_mapping, int T, int H, int D, int P,
                       int64_t num_pages)
{
    for (int t = 0; t < T; t++) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_pages * (int64_t)P)
            return ORC_ERR_INDEX;
        int64_t page = slot / P;
        int64_t off = slot % P;
        for (int h = 0; h < H; h++) {
            for (int d = 0; d < D; d++) {
                float x = orc_bf16_to_f32(x_new[((int64_t)t * H + h) * D + d]);
                float y = x / head_scales[h];
                cache[((page * H + h) * P + off) * D + d] = orc_e4m3_encode(y);
            }
        }
    }
    return ORC_OK;
}

/* Append with one scale per (token, KV head) row, computed from the row and
 * stored beside it in scales [num_pages][H][P]. */
int orc_kv_append_token(const uint16_t *x_new, uint8_t *cache, float *scales,
                        const int64_t *slot_mapping, int T, int H, int D, int P,
                        int64_t num_pages)
{
    for (int t = 0; t < T; t++) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_pages * (int64_t)P)
            return ORC_ERR_INDEX;
        int64_t page = slot / P;
        int64_t off = slot % P;
        for (int h = 0; h < H; h++) {
            const uint16_t *row = x_new + ((int64_t)t * H + h) * D;
            int64_t crow = (page * H + h) * P + off;
            float amax = 0.0f;
            for (int d = 0; d < D; d++) {
                float a = fabsf(orc_bf16_to_f32(row[d]));
                if (a > amax)
                    amax = a;
            }
            float s = amax / 448.0f;
            scales[crow] = s;
            for (int d = 0; d < D; d++) {
                float x = orc_bf16_to_f32(row[d]);
                cache[crow * D + d] = (s == 0.0f) ? 0 : orc_e4m3_encode(x / s);
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Dequantised element of a cache row ([FP8]: converted when read). */
static double cache_elem(const void *cache, int cache_dtype, int64_t idx, double scale)
{
    if (cache_dtype == ORC_CACHE_BF16)
        return (double)orc_bf16_to_f32(((const uint16_t *)cache)[idx]) * scale;
    return orc_e4m3_value(((const uint8_t *)cache)[idx]) * scale;
}

/* Resolve logical token t of one request to its cache row index ([PAGE]):
 * page = block_table[t / P], offset = t % P; returns -1 for a bad page id. */
static int64_t token_row(const int32_t *bt_row, int64_t t, int P, int64_t num_pages)
{
    int32_t page = bt_row[t / P];
    if (page < 0 || page >= num_pages)
        return -1;
    return (int64_t)page * P + (t % P);
}

/* Decode attention for one query head of one request over its whole context
 * (GQA/MHA).  Plain definition:
 *   s_t = softmax_scale * sum_d q_d * (dequant(K[t][d]) )      t = 0..L-1
 *   p_t = exp(s_t - max_t s_t),  out_d = sum_t p_t dequant(V[t][d]) / sum_t p_t
 *   lse = max_t s_t + log(sum_t p_t)
 * with K/V rows found through the block table ([PAGE]) in the KV head kvh that
 * serves this query head.  L == 0 gives out = 0 and lse = -inf. */
int orc_paged_decode_one(double *out, double *lse, const uint16_t *q,
                         const void *k_cache, const void *v_cache, int cache_dtype,
                         const int32_t *bt_row, int L, int Hkv, int kvh, int D, int P,
                         int64_t num_pages, float k_scale, float v_scale, float softmax_scale)
{
    for (int d = 0; d < D; d++)
        out[d] = 0.0;
    if (L <= 0) {
        *lse = -INFINITY;
        return ORC_OK;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    if (!s)
        return ORC_ERR_NOMEM;
    for (int64_t t = 0; t < L; t++) {
        int64_t row = token_row(bt_row, t, P, num_pages);
        if (row < 0) {
            free(s);
            return ORC_ERR_INDEX;
        }
        int64_t base = ((row / P) * Hkv + kvh) * (int64_t)P * D + (row % P) * D;
        double acc = 0.0;
        for (int d = 0; d < D; d++)
            acc += (double)orc_bf16_to_f32(q[d]) * cache_elem(k_cache, cache_dtype, base + d, k_scale);
        s[t] = (double)softmax_scale * acc;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < L; t++)
        if (s[t] > m)
            m = s[t];
    double l = 0.0;
    for (int64_t t = 0; t < L; t++) {
        double p = exp(s[t] - m);
        int64_t row = token_row(bt_row, t, P, num_pages);
        int64_t base = ((row / P) * Hkv + kvh) * (int64_t)P * D + (row % P) * D;
        l += p;
        for (int d = 0; d < D; d++)
            out[d] += p * cache_elem(v_cache, cache_dtype, base + d, v_scale);
    }
    for (int d = 0; d < D; d++)
        out[d] /= l;
    *lse = m + log(l);
    free(s);
    return ORC_OK;
}

/* Whole batch: out [B][Hq][D], lse [B][Hq] (lse may be NULL); query head h reads
 * KV head h / (Hq / Hkv).  Units u = b * Hq + h in [u_begin, u_end) only, so that
 * a caller can split the batch over threads without changing any arithmetic. */
int orc_paged_decode(double *out, double *lse, const uint16_t *q,
                     const void *k_cache, const void *v_cache, int cache_dtype,
                     const int32_t *block_tables, int max_pages_per_seq,
                     const int32_t *context_lens, int B, int Hq, int Hkv, int D, int P,
                     int64_t num_pages, float k_scale, float v_scale, float softmax_scale,
                     int64_t u_begin, int64_t u_end)
{
    if (Hkv <= 0 || Hq % Hkv != 0)
        return ORC_ERR_ARG;
    int G = Hq / Hkv;
    if (u_end > (int64_t)B * Hq)
        u_end = (int64_t)B * Hq;
    for (int64_t u = u_begin; u < u_end; u++) {
        int b = (int)(u / Hq), h = (int)(u % Hq);
        int L = context_lens[b];
        if (L > max_pages_per_seq * P)
            return ORC_ERR_INDEX;
        double lse_bh;
        int rc = orc_paged_decode_one(out + u * D, &lse_bh, q + u * D, k_cache, v_cache,
                                      cache_dtype, block_tables + (int64_t)b * max_pages_per_seq,
                                      L, Hkv, h / G, D, P, num_pages, k_scale, v_scale,
                                      softmax_scale);
        if (rc != ORC_OK)
            return rc;
        if (lse)
            lse[u] = lse_bh;
    }
    return ORC_OK;
}

/* Decode attention as orc_paged_decode_one with an e4m3 cache whose elements
 * are dequantised with the scale of their granularity ([SCL]):
 *   K(t)[d] = e4m3(Kcode) * ks(t),  V(t)[d] = e4m3(Vcode) * vs(t)
 * where ks/vs pick scales[0], scales[kvh] or the token row's own scale. */
int orc_paged_decode_scaled_one(double *out, double *lse, const uint16_t *q,
                                const uint8_t *k_cache, const uint8_t *v_cache, int granularity,
                                const float *k_scales, const float *v_scales,
                                const int32_t *bt_row, int L, int Hkv, int kvh, int D, int P,
                                int64_t num_pages, float softmax_scale)
{
    for (int d = 0; d < D; d++)
        out[d] = 0.0;
    if (L <= 0) {
        *lse = -INFINITY;
        return ORC_OK;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    if (!s)
        return ORC_ERR_NOMEM;
    for (int64_t t = 0; t < L; t++) {
        int64_t row = token_row(bt_row, t, P, num_pages);
        if (row < 0) {
            free(s);
            return ORC_ERR_INDEX;
        }
        int64_t crow = ((row / P) * Hkv + kvh) * (int64_t)P + row % P;
        double ks = scale_at(granularity, k_scales, crow, kvh);
        double acc = 0.0;
        for (int d = 0; d < D; d++)
            acc += (double)orc_bf16_to_f32(q[d]) * (orc_e4m3_value(k_cache[crow * D + d]) * ks);
        s[t] = (double)softmax_scale * acc;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < L; t++)
        if (s[t] > m)
            m = s[t];
    double l = 0.0;
    for (int64_t t = 0; t < L; t++) {
        double p = exp(s[t] - m);
        int64_t row = token_row(bt_row, t, P, num_pages);
        int64_t crow = ((row / P) * Hkv + kvh) * (int64_t)P + row % P;
        double vs = scale_at(granularity, v_scales, crow, kvh);
        l += p;
        for (int d = 0; d < D; d++)
            out[d] += p * (orc_e4m3_value(v_cache[crow * D + d]) * vs);
    }
    for (int d = 0; d < D; d++)
        out[d] /= l;
    *lse = m + log(l);
    free(s);
    return ORC_OK;
}

/* Whole batch of orc_paged_decode_scaled_one, units [u_begin, u_end) as in
 * orc_paged_decode. */
int orc_paged_decode_scaled(double *out, double *lse, const uint16_t *q, const uint8_t *k_cache,
                            const uint8_t *v_cache, int granularity, const float *k_scales,
                            const float *v_scales, const int32_t *block_tables,
                            int max_pages_per_seq, const int32_t *context_lens, int B, int Hq,
                            int Hkv, int D, int P, int64_t num_pages, float softmax_scale,
                            int64_t u_begin, int64_t u_end)
{
    if (Hkv <= 0 || Hq % Hkv != 0)
        return ORC_ERR_ARG;
    if (granularity != ORC_SCALE_TENSOR && granularity != ORC_SCALE_HEAD &&
        granularity != ORC_SCALE_TOKEN)
        return ORC_ERR_ARG;
    int G = Hq / Hkv;
    if (u_end > (int64_t)B * Hq)
        u_end = (int64_t)B * Hq;
    for (int64_t u = u_begin; u < u_end; u++) {
        int b = (int)(u / Hq), h = (int)(u % Hq);
        int L = context_lens[b];
        if (L > max_pages_per_seq * P)
            return ORC_ERR_INDEX;
        double lse_bh;
        int rc = orc_paged_decode_scaled_one(out + u * D, &lse_bh, q + u * D, k_cache, v_cache,
                                             granularity, k_scales, v_scales,
                                             block_tables + (int64_t)b * max_pages_per_seq, L,
                                             Hkv, h / G, D, P, num_pages, softmax_scale);
        if (rc != ORC_OK)
            return rc;
        if (lse)
            lse[u] = lse_bh;
    }
    return ORC_OK;
}

/* Several new query tokens per request ([CHK] chunked prefill / [SPEC]
 * verification): request b's last n_b = q_start[b+1] - q_start[b] positions,
 * L_b - n_b .. L_b - 1, are queries; query i sits at position L_b - n_b + i and
 * attends the keys 0 .. L_b - n_b + i (causal within the new tokens).  That is
 * decode attention (orc_paged_decode_one) over a context of L_b - n_b + i + 1
 * tokens.  q / out rows are [q_start[b] + i][Hq][D]; lse [q_start[b] + i][Hq]. */
int orc_paged_prefill(double *out, double *lse, const uint16_t *q, const void *k_cache,
                      const void *v_cache, int cache_dtype, const int32_t *block_tables,
                      int max_pages_per_seq, const int32_t *context_lens, const int32_t *q_start,
                      int B, int Hq, int Hkv, int D, int P, int64_t num_pages, float k_scale,
                      float v_scale, float softmax_scale, int64_t r_begin, int64_t r_end)
{
    if (Hkv <= 0 || Hq % Hkv != 0)
        return ORC_ERR_ARG;
    int G = Hq / Hkv;
    int64_t total = q_start[B];
    if (r_end > total * Hq)
        r_end = total * Hq;
    for (int64_t u = r_begin; u < r_end; u++) {
        int64_t row = u / Hq; /* query token row in q */
        int h = (int)(u % Hq);
        int b = 0;
        while (q_start[b + 1] <= row)
            b++;
        int n = q_start[b + 1] - q_start[b];
        int L = context_lens[b];
        int i = (int)(row - q_start[b]);
        if (n > L || L > max_pages_per_seq * P)
            return ORC_ERR_INDEX;
        double lse_r;
        int rc = orc_paged_decode_one(out + u * D, &lse_r, q + u * D, k_cache, v_cache, cache_dtype,
                                      block_tables + (int64_t)b * max_pages_per_seq, L - n + i + 1,
                                      Hkv, h / G, D, P, num_pages, k_scale, v_scale, softmax_scale);
        if (rc != ORC_OK)
            return rc;
        if (lse)
            lse[u] = lse_r;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Split-KV form ([OSM]): the context is cut into chunks of `chunk` tokens; each
 * chunk c yields its own state (m_c, l_c, o_c) with
 *   m_c = max_{t in c} s_t,  l_c = sum_{t in c} exp(s_t - m_c),
 *   o_c = sum_{t in c} exp(s_t - m_c) v_t,
 * and the states are merged by the log-sum-exp rule
 *   M = max_c m_c,  out = sum_c e^{m_c - M} o_c / sum_c e^{m_c - M} l_c.
 * The result must equal orc_paged_decode_one (the pages' claim that blockwise
 * attention gives the same numbers as full attention). */
int orc_paged_decode_split_one(double *out, double *lse, const uint16_t *q,
                               const void *k_cache, const void *v_cache, int cache_dtype,
                               const int32_t *bt_row, int L, int Hkv, int kvh, int D, int P,
                               int64_t num_pages, float k_scale, float v_scale,
                               float softmax_scale, int chunk)
{
    if (chunk <= 0)
        return ORC_ERR_ARG;
    for (int d = 0; d < D; d++)
        out[d] = 0.0;
    if (L <= 0) {
        *lse = -INFINITY;
        return ORC_OK;
    }
    int nc = (L + chunk - 1) / chunk;
    double *m = (double *)malloc(sizeof(double) * (size_t)nc);
    double *l = (double *)malloc(sizeof(double) * (size_t)nc);
    double *o = (double *)calloc((size_t)nc * (size_t)D, sizeof(double));
    double *s = (double *)malloc(sizeof(double) * (size_t)chunk);
    if (!m || !l || !o || !s) {
        free(m); free(l); free(o); free(s);
        return ORC_ERR_NOMEM;
    }
    int rc = ORC_OK;
    for (int c = 0; c < nc && rc == ORC_OK; c++) {
        int64_t t0 = (int64_t)c * chunk;
        int64_t t1 = t0 + chunk < L ? t0 + chunk : L;
        m[c] = -INFINITY;
        for (int64_t t = t0; t < t1; t++) {
            int64_t row = token_row(bt_row, t, P, num_pages);
            if (row < 0) {
                rc = ORC_ERR_INDEX;
                break;
            }
            int64_t base = ((row / P) * Hkv + kvh) * (int64_t)P * D + (row % P) * D;
            double acc = 0.0;
            for (int d = 0; d < D; d++)
                acc += (double)orc_bf16_to_f32(q[d]) * cache_elem(k_cache, cache_dtype, base + d, k_scale);
            s[t - t0] = (double)softmax_scale * acc;
            if (s[t - t0] > m[c])
                m[c] = s[t - t0];
        }
        if (rc != ORC_OK)
            break;
        l[c] = 0.0;
        for (int64_t t = t0; t < t1; t++) {
            double p = exp(s[t - t0] - m[c]);
            int64_t row = token_row(bt_row, t, P, num_pages);
            int64_t base = ((row / P) * Hkv + kvh) * (int64_t)P * D + (row % P) * D;
            l[c] += p;
            for (int d = 0; d < D; d++)
                o[(int64_t)c * D + d] += p * cache_elem(v_cache, cache_dtype, base + d, v_scale);
        }
    }
    if (rc == ORC_OK) {
        double M = -INFINITY;
        for (int c = 0; c < nc; c++)
            if (m[c] > M)
                M = m[c];
        double den = 0.0;
        for (int c = 0; c < nc; c++) {
            double w = exp(m[c] - M);
            den += w * l[c];
            for (int d = 0; d < D; d++)
                out[d] += w * o[(int64_t)c * D + d];
        }
        for (int d = 0; d < D; d++)
            out[d] /= den;
        *lse = M + log(den);
    }
    free(m); free(l); free(o); free(s);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* MLA absorbed-latent decode for one head of one request ([MLA]).  Every token
 * has one latent row c_t of width Dqk (latent + rope part) shared by all heads,
 * stored e4m3 in pages of P rows: cache [num_pages][P][Dqk].  The absorbed
 * reading uses the whole row as the key and its first Dv entries as the value:
 *   s_t = softmax_scale * sum_{d<Dqk} q_d * c_t[d] * ckv_scale
 *   out = sum_t p_t c_t[0:Dv] * ckv_scale / sum_t p_t
 * over t in the top-k list (entries < 0 are padding and skipped), or over all
 * t < L when topk is NULL.  A listed t >= L, or a bad page id, is an error. */
int orc_mla_decode_one(double *out, double *lse, const uint16_t *q, const uint8_t *ckv_cache,
                       const int32_t *bt_row, int L, const int32_t *topk, int topk_n, int Dqk,
                       int Dv, int P, int64_t num_pages, float ckv_scale, float softmax_scale)
{
    for (int d = 0; d < Dv; d++)
        out[d] = 0.0;
    int n = topk ? topk_n : L;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!s || !rows) {
        free(s); free(rows);
        return ORC_ERR_NOMEM;
    }
    int cnt = 0;
    for (int j = 0; j < n; j++) {
        int64_t t = topk ? topk[j] : j;
        if (t < 0)
            continue;
        if (t >= L) {
            free(s); free(rows);
            return ORC_ERR_INDEX;
        }
        int64_t row = token_row(bt_row, t, P, num_pages);
        if (row < 0) {
            free(s); free(rows);
            return ORC_ERR_INDEX;
        }
        double acc = 0.0;
        for (int d = 0; d < Dqk; d++)
            acc += (double)orc_bf16_to_f32(q[d]) * orc_e4m3_value(ckv_cache[row * Dqk + d]) * (double)ckv_scale;
        s[cnt] = (double)softmax_scale * acc;
        rows[cnt] = row;
        cnt++;
    }
    if (cnt == 0) {
        *lse = -INFINITY;
        free(s); free(rows);
        return ORC_OK;
    }
    double m = -INFINITY;
    for (int j = 0; j < cnt; j++)
        if (s[j] > m)
            m = s[j];
    double l = 0.0;
    for (int j = 0; j < cnt; j++) {
        double p = exp(s[j] - m);
        l += p;
        for (int d = 0; d < Dv; d++)
            out[d] += p * orc_e4m3_value(ckv_cache[rows[j] * Dqk + d]) * (double)ckv_scale;
    }
    for (int d = 0; d < Dv; d++)
        out[d] /= l;
    *lse = m + log(l);
    free(s); free(rows);
    return ORC_OK;
}

/* Whole batch for MLA: out [B][H][Dv], lse [B][H] (may be NULL), q [B][H][Dqk],
 * topk [B][topk_n] or NULL.  Units u = b * H + h in [u_begin, u_end). */
int orc_mla_decode(double *out, double *lse, const uint16_t *q, const uint8_t *ckv_cache,
                   const int32_t *block_tables, int max_pages_per_seq, const int32_t *context_lens,
                   const int32_t *topk, int topk_n, int B, int H, int Dqk, int Dv, int P,
                   int64_t num_pages, float ckv_scale, float softmax_scale,
                   int64_t u_begin, int64_t u_end)
{
    if (u_end > (int64_t)B * H)
        u_end = (int64_t)B * H;
    for (int64_t u = u_begin; u < u_end; u++) {
        int b = (int)(u / H);
        int L = context_lens[b];
        if (L > max_pages_per_seq * P)
            return ORC_ERR_INDEX;
        double lse_bh;
        int rc = orc_mla_decode_one(out + u * Dv, &lse_bh, q + u * Dqk, ckv_cache,
                                    block_tables + (int64_t)b * max_pages_per_seq, L,
                                    topk ? topk + (int64_t)b * topk_n : NULL, topk_n, Dqk, Dv, P,
                                    num_pages, ckv_scale, softmax_scale);
        if (rc != ORC_OK)
            return rc;
        if (lse)
            lse[u] = lse_bh;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* KV bytes of a cache ([KVB]): 2 (K and V) x layers x KV heads x head_dim x
 * tokens x bytes per element. */
int64_t orc_kv_bytes(int64_t layers, int64_t kv_heads, int64_t head_dim, int64_t tokens,
                     int64_t bytes_per_elem)
{
    return 2 * layers * kv_heads * head_dim * tokens * bytes_per_elem;
}

/* ------------------------------------------------------------------------- */
/* KV page integrity check (Workers AI post, section 3 "共用 KV キャッシュの保護",
 * 動作原理): every physical page has a tag that changes whenever the page is
 * handed out again; before decode, each request's pages are compared with the
 * tags it recorded when it mapped them.  The request reads the entries
 * i < ceil(L / P) of its block-table row.  status[b] = 0, or the OR of
 * ORC_REQ_TAG_MISMATCH (a read page now carries another tag) and
 * ORC_REQ_BAD_INDEX (a read entry outside [0, num_pages), or L outside
 * [0, max_pages * P]; then the row is checked up to the clamped length). */
int orc_verify_page_tags(const int32_t *block_tables, const uint32_t *table_tags, int max_pages,
                         const int32_t *context_lens, int B, int P, const uint32_t *page_tags,
                         int64_t num_pages, int32_t *status)
{
    if (B < 0 || max_pages <= 0 || P <= 0 || num_pages <= 0)
        return ORC_ERR_ARG;
    for (int b = 0; b < B; b++) {
        int32_t flags = 0;
        int64_t L = context_lens[b];
        if (L < 0) {
            flags |= ORC_REQ_BAD_INDEX;
            L = 0;
        } else if (L > (int64_t)max_pages * P) {
            flags |= ORC_REQ_BAD_INDEX;
            L = (int64_t)max_pages * P;
        }
        int64_t used = (L + P - 1) / P;
        for (int64_t i = 0; i < used; i++) {
            int32_t page = block_tables[(int64_t)b * max_pages + i];
            if (page < 0 || page >= num_pages)
                flags |= ORC_REQ_BAD_INDEX;
            else if (page_tags[page] != table_tags[(int64_t)b * max_pages + i])
                flags |= ORC_REQ_TAG_MISMATCH;
        }
        status[b] = flags;
    }
    return ORC_OK;
}
