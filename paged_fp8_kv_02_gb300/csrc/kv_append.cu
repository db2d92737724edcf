// kv_append.cu -- quantise new bf16 K/V rows (or MLA latent rows) to e4m3 and
// scatter them into pages through a slot mapping.
//
// Workers AI post (より小さく、高速で、安全に), §1 "KV キャッシュの量子化": the
// cache holds 8-bit e4m3 instead of BF16.  Inference-engine scheduling
// explainer (推論エンジンの実践), "FP8 KV のエンジニアリング上の制約": the scale
// is per tensor, per head or per token; "PagedAttention の 2 つの原語": rows go
// to fixed-size pages.
//
// Per-tensor and per-head scales: one thread handles 16 consecutive elements
// of one (token, head) row: two 16-byte bf16 loads, 16 IEEE fp32 divisions
// (correctly rounded, matching the definition code = e4m3(fp32(x) / scale)),
// eight cvt.rn.satfinite.e4m3x2 and one 16-byte store.  Per-token scales: one
// warp per row, lane c holding elements 16c..16c+15; a warp max gives the
// row's amax, the scale amax / 448 is stored beside the row and the same
// divisions follow.  The step is tiny (a few hundred KB per decode step) and
// latency-bound; its grid covers K and V in one launch.
#include <cuda_bf16.h>

#include "pfkv_internal.h"
#include "pfkv_ptx.cuh"

namespace pfkv {
namespace {

struct AppendArgs {
  const uint16_t* x[2];  // K, V sources (bf16 bits) [T][H][D]
  void* cache[2];        // destinations [pages][H][P][D]
  float scale[2];
  const float* dscale[2];  // device scales (per tensor or per head), or null
  int dscale_stride;       // 1: indexed by head; 0: one scale for all heads
  float* tscale[2];        // per-token scales written beside each row
  const int64_t* slots;
  int T, H, D, P;
  int64_t num_pages;
};

template <bool kFp8, bool kDevScale>
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendArgs a) {
  const int which = blockIdx.y;
  const int chunks = a.D >> 4;  // 16-element chunks per row
  const int64_t n = (int64_t)a.T * a.H * chunks;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int c = (int)(i % chunks);
  const int64_t th = i / chunks;  // t * H + h
  const int h = (int)(th % a.H);
  const int t = (int)(th / a.H);
  const int64_t slot = a.slots[t];
  if (slot < 0 || slot >= a.num_pages * a.P) return;  // skipped; validate_tables reports
  const int64_t page = slot / a.P;
  const int off = (int)(slot - page * a.P);
  const int64_t dst = ((page * a.H + h) * a.P + off) * a.D + (int64_t)c * 16;
  const uint16_t* xs = which ? a.x[1] : a.x[0];
  void* cache = which ? a.cache[1] : a.cache[0];
  const uint4* src = reinterpret_cast<const uint4*>(xs + th * a.D + (int64_t)c * 16);
  const uint4 lo = src[0], hi = src[1];
  if constexpr (kFp8) {
    float s;
    if constexpr (kDevScale)
      s = __ldg((which ? a.dscale[1] : a.dscale[0]) + (int64_t)h * a.dscale_stride);
    else
      s = which ? a.scale[1] : a.scale[0];
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t packed[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t q0 = w[2 * k], q1 = w[2 * k + 1];
      const uint16_t e01 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(q0), s), __fdiv_rn(bf16_hi(q0), s));
      const uint16_t e23 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(q1), s), __fdiv_rn(bf16_hi(q1), s));
      packed[k] = (uint32_t)e01 | ((uint32_t)e23 << 16);
    }
    *reinterpret_cast<uint4*>(static_cast<uint8_t*>(cache) + dst) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
  } else {
    uint4* d = reinterpret_cast<uint4*>(static_cast<uint16_t*>(cache) + dst);
    d[0] = lo;
    d[1] = hi;
  }
}

// Per-token scales: warp w of the block quantises row (token, head) number
// 8 * blockIdx.x + w.  D <= 512, so each lane holds at most one 16-element chunk.
__global__ void __launch_bounds__(256) kv_append_token_kernel(const AppendArgs a) {
  const int which = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int64_t th = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // t * H + h
  if (th >= (int64_t)a.T * a.H) return;
  const int h = (int)(th % a.H);
  const int t = (int)(th / a.H);
  const int64_t slot = a.slots[t];
  if (slot < 0 || slot >= a.num_pages * a.P) return;  // skipped; validate_tables reports
  const int64_t page = slot / a.P;
  const int off = (int)(slot - page * a.P);
  const int64_t row = (page * a.H + h) * a.P + off;
  const int chunks = a.D >> 4;
  const bool mine = lane < chunks;
  uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (mine) {
    const uint4* src = reinterpret_cast<const uint4*>((which ? a.x[1] : a.x[0]) + th * a.D + lane * 16);
    const uint4 lo = src[0], hi = src[1];
    w[0] = lo.x, w[1] = lo.y, w[2] = lo.z, w[3] = lo.w, w[4] = hi.x, w[5] = hi.y, w[6] = hi.z, w[7] = hi.w;
  }
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  const float s = __fdiv_rn(m, 448.f);
  if (lane == 0) (which ? a.tscale[1] : a.tscale[0])[row] = s;
  if (!mine) return;
  uint32_t packed[4] = {0, 0, 0, 0};
  if (s != 0.f) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t q0 = w[2 * k], q1 = w[2 * k + 1];
      const uint16_t e01 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(q0), s), __fdiv_rn(bf16_hi(q0), s));
      const uint16_t e23 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(q1), s), __fdiv_rn(bf16_hi(q1), s));
      packed[k] = (uint32_t)e01 | ((uint32_t)e23 << 16);
    }
  }
  *reinterpret_cast<uint4*>(static_cast<uint8_t*>(which ? a.cache[1] : a.cache[0]) + row * a.D + lane * 16) =
      make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

// gran < 0: host scalar scales; otherwise a pfkv_scale_granularity with
// device scale arrays (read for TENSOR/HEAD, written for TOKEN).
int append_common(bool fp8, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                  const int64_t* slot_mapping, int T, int H, int D, int P, int64_t num_pages,
                  float k_scale, float v_scale, int gran, float* k_scales, float* v_scales,
                  cudaStream_t stream) {
  clear_error();
  if (T < 0 || H <= 0 || D <= 0 || P <= 0 || num_pages <= 0)
    return fail(PFKV_ERR_INVALID_ARG, "kv_append: bad sizes T=%d H=%d D=%d P=%d pages=%lld", T, H,
                D, P, (long long)num_pages);
  if (D % 16 != 0) return fail(PFKV_ERR_UNSUPPORTED, "kv_append: head_dim %d not a multiple of 16", D);
  if (T == 0) return PFKV_OK;
  if (!k_new || !k_cache || !slot_mapping)
    return fail(PFKV_ERR_INVALID_ARG, "kv_append: null K/slot pointer");
  const bool has_v = (v_new != nullptr) || (v_cache != nullptr);
  if (has_v && (!v_new || !v_cache))
    return fail(PFKV_ERR_INVALID_ARG, "kv_append: v_new and v_cache must both be set or both NULL");
  if (fp8 && gran < 0) {
    if (!(k_scale > 0.f) || !isfinite(k_scale) || (has_v && (!(v_scale > 0.f) || !isfinite(v_scale))))
      return fail(PFKV_ERR_INVALID_ARG, "kv_append_fp8: scales must be finite and > 0");
  }
  if (gran >= 0) {
    if (gran != PFKV_SCALE_TENSOR && gran != PFKV_SCALE_HEAD && gran != PFKV_SCALE_TOKEN)
      return fail(PFKV_ERR_INVALID_ARG, "kv_append_fp8_scaled: unknown granularity %d", gran);
    if (!k_scales || (has_v && !v_scales))
      return fail(PFKV_ERR_INVALID_ARG, "kv_append_fp8_scaled: null scale array");
    if (!aligned(k_scales, 4) || (has_v && !aligned(v_scales, 4)))
      return fail(PFKV_ERR_INVALID_ARG, "kv_append_fp8_scaled: scale arrays must be 4-byte aligned");
    if (gran == PFKV_SCALE_TOKEN && D > 512)
      return fail(PFKV_ERR_UNSUPPORTED, "kv_append_fp8_scaled: per-token scales need head_dim <= 512");
  }
  if (!aligned(k_new, 16) || !aligned(k_cache, 16) || (has_v && (!aligned(v_new, 16) || !aligned(v_cache, 16))) ||
      !aligned(slot_mapping, 8))
    return fail(PFKV_ERR_INVALID_ARG, "kv_append: pointers must be 16-byte aligned");
  AppendArgs a;
  a.x[0] = static_cast<const uint16_t*>(k_new);
  a.x[1] = static_cast<const uint16_t*>(v_new);
  a.cache[0] = k_cache;
  a.cache[1] = v_cache;
  a.scale[0] = k_scale;
  a.scale[1] = v_scale;
  a.dscale[0] = k_scales;
  a.dscale[1] = v_scales;
  a.dscale_stride = gran == PFKV_SCALE_HEAD ? 1 : 0;
  a.tscale[0] = k_scales;
  a.tscale[1] = v_scales;
  a.slots = slot_mapping;
  a.T = T;
  a.H = H;
  a.D = D;
  a.P = P;
  a.num_pages = num_pages;
  if (gran == PFKV_SCALE_TOKEN) {
    const int64_t blocks = ((int64_t)T * H + 7) / 8;
    if (blocks > 0x7FFFFFFF) return fail(PFKV_ERR_UNSUPPORTED, "kv_append: too many tokens");
    kv_append_token_kernel<<<dim3((unsigned)blocks, has_v ? 2 : 1), 256, 0, stream>>>(a);
    return check_cuda("kv_append launch");
  }
  const int64_t n = (int64_t)T * H * (D / 16);
  const int64_t blocks = (n + 255) / 256;
  if (blocks > 0x7FFFFFFF) return fail(PFKV_ERR_UNSUPPORTED, "kv_append: too many tokens");
  dim3 grid((unsigned)blocks, has_v ? 2 : 1);
  if (fp8 && gran >= 0)
    kv_append_kernel<true, true><<<grid, 256, 0, stream>>>(a);
  else if (fp8)
    kv_append_kernel<true, false><<<grid, 256, 0, stream>>>(a);
  else
    kv_append_kernel<false, false><<<grid, 256, 0, stream>>>(a);
  return check_cuda("kv_append launch");
}

}  // namespace
}  // namespace pfkv

extern "C" {

int pfkv_kv_append_fp8(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                       const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                       int page_size, int64_t num_pages, float k_scale, float v_scale,
                       pfkv_stream_t stream) {
  return pfkv::append_common(true, k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens,
                             num_kv_heads, head_dim, page_size, num_pages, k_scale, v_scale, -1,
                             nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int pfkv_kv_append_fp8_scaled(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                              const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                              int head_dim, int page_size, int64_t num_pages,
                              pfkv_scale_granularity granularity, float* k_scales, float* v_scales,
                              pfkv_stream_t stream) {
  return pfkv::append_common(true, k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens,
                             num_kv_heads, head_dim, page_size, num_pages, 1.f, 1.f,
                             (int)granularity, k_scales, v_scales,
                             reinterpret_cast<cudaStream_t>(stream));
}

int pfkv_kv_append_bf16(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                        const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                        int page_size, int64_t num_pages, pfkv_stream_t stream) {
  return pfkv::append_common(false, k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens,
                             num_kv_heads, head_dim, page_size, num_pages, 1.f, 1.f, -1, nullptr,
                             nullptr, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
