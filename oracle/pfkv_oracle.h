/*
 * pfkv_oracle.h -- CPU oracle for paged FP8 (e4m3) KV decode attention.
 * TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU-baseline leg of the
 * benchmark).  See pfkv_oracle.c for the definitions each function follows.
 */
#ifndef PFKV_ORACLE_H
#define PFKV_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_ERR_ARG = -1, ORC_ERR_INDEX = -4, ORC_ERR_NOMEM = -5 };
enum { ORC_CACHE_FP8_E4M3 = 0, ORC_CACHE_BF16 = 1 };
enum { ORC_SCALE_TENSOR = 0, ORC_SCALE_HEAD = 1, ORC_SCALE_TOKEN = 2 };

double orc_e4m3_value(uint8_t code);
uint8_t orc_e4m3_encode(float x);
void orc_e4m3_encode_array(const float *x, uint8_t *out, int64_t n);
float orc_bf16_to_f32(uint16_t b);

int orc_kv_append(const uint16_t *x_new, uint8_t *cache, const int64_t *slot_mapping,
                  int T, int H, int D, int P, int64_t num_pages, float scale);
int orc_kv_append_bf16(const uint16_t *x_new, uint16_t *cache, const int64_t *slot_mapping,
                       int T, int H, int D, int P, int64_t num_pages);
int orc_kv_append_head(const uint16_t *x_new, uint8_t *cache, const float *head_scales,
                       const int64_t *slot_mapping, int T, int H, int D, int P,
                       int64_t num_pages);
int orc_kv_append_token(const uint16_t *x_new, uint8_t *cache, float *scales,
                        const int64_t *slot_mapping, int T, int H, int D, int P,
                        int64_t num_pages);

int orc_paged_decode_one(double *out, double *lse, const uint16_t *q,
                         const void *k_cache, const void *v_cache, int cache_dtype,
                         const int32_t *bt_row, int L, int Hkv, int kvh, int D, int P,
                         int64_t num_pages, float k_scale, float v_scale, float softmax_scale);
int orc_paged_decode(double *out, double *lse, const uint16_t *q,
                     const void *k_cache, const void *v_cache, int cache_dtype,
                     const int32_t *block_tables, int max_pages_per_seq,
                     const int32_t *context_lens, int B, int Hq, int Hkv, int D, int P,
                     int64_t num_pages, float k_scale, float v_scale, float softmax_scale,
                     int64_t u_begin, int64_t u_end);
int orc_paged_decode_scaled_one(double *out, double *lse, const uint16_t *q,
                                const uint8_t *k_cache, const uint8_t *v_cache, int granularity,
                                const float *k_scales, const float *v_scales,
                                const int32_t *bt_row, int L, int Hkv, int kvh, int D, int P,
                                int64_t num_pages, float softmax_scale);
int orc_paged_decode_scaled(double *out, double *lse, const uint16_t *q, const uint8_t *k_cache,
                            const uint8_t *v_cache, int granularity, const float *k_scales,
                            const float *v_scales, const int32_t *block_tables,
                            int max_pages_per_seq, const int32_t *context_lens, int B, int Hq,
                            int Hkv, int D, int P, int64_t num_pages, float softmax_scale,
                            int64_t u_begin, int64_t u_end);
int orc_paged_prefill(double *out, double *lse, const uint16_t *q, const void *k_cache,
                      const void *v_cache, int cache_dtype, const int32_t *block_tables,
                      int max_pages_per_seq, const int32_t *context_lens, const int32_t *q_start,
                      int B, int Hq, int Hkv, int D, int P, int64_t num_pages, float k_scale,
                      float v_scale, float softmax_scale, int64_t r_begin, int64_t r_end);
int orc_paged_decode_split_one(double *out, double *lse, const uint16_t *q,
                               const void *k_cache, const void *v_cache, int cache_dtype,
                               const int32_t *bt_row, int L, int Hkv, int kvh, int D, int P,
                               int64_t num_pages, float k_scale, float v_scale,
                               float softmax_scale, int chunk);

int orc_mla_decode_one(double *out, double *lse, const uint16_t *q, const uint8_t *ckv_cache,
                       const int32_t *bt_row, int L, const int32_t *topk, int topk_n, int Dqk,
                       int Dv, int P, int64_t num_pages, float ckv_scale, float softmax_scale);
int orc_mla_decode(double *out, double *lse, const uint16_t *q, const uint8_t *ckv_cache,
                   const int32_t *block_tables, int max_pages_per_seq, const int32_t *context_lens,
                   const int32_t *topk, int topk_n, int B, int H, int Dqk, int Dv, int P,
                   int64_t num_pages, float ckv_scale, float softmax_scale,
                   int64_t u_begin, int64_t u_end);

#define ORC_REQ_TAG_MISMATCH 0x1
#define ORC_REQ_BAD_INDEX 0x2
int orc_verify_page_tags(const int32_t *block_tables, const uint32_t *table_tags, int max_pages,
                         const int32_t *context_lens, int B, int P, const uint32_t *page_tags,
                         int64_t num_pages, int32_t *status);
int64_t orc_kv_bytes(int64_t layers, int64_t kv_heads, int64_t head_dim, int64_t tokens,
                     int64_t bytes_per_elem);

#ifdef __cplusplus
}
#endif
#endif
