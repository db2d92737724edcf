// kv_append.cu -- quantise new bf16 K/V rows (or MLA latent rows) to e4m3 with
// a per-tensor fp32 scale and scatter them into pages through a slot mapping.
//
// Workers AI post (より小さく、高速で、安全に), §1 "KV キャッシュの量子化": the
// cache holds 8-bit e4m3 instead of BF16.  Inference-engine scheduling
// explainer (推論エンジンの実践), "FP8 KV のエンジニアリング上の制約": one scale
// per tensor here; "PagedAttention の 2 つの原語": rows go to fixed-size pages.
//
// One thread handles 16 consecutive elements of one (token, head) row: two
// 16-byte bf16 loads, 16 IEEE fp32 divisions (correctly rounded, matching the
// definition code = e4m3(fp32(x) / scale)), eight cvt.rn.satfinite.e4m3x2 and
// one 16-byte store.  The step is tiny (a few hundred KB per decode step) and
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
  const int64_t* slots;
  int T, H, D, P;
  int64_t num_pages;
};

template <bool kFp8>
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
    const float s = which ? a.scale[1] : a.scale[0];
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

int append_common(bool fp8, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                  const int64_t* slot_mapping, int T, int H, int D, int P, int64_t num_pages,
                  float k_scale, float v_scale, cudaStream_t stream) {
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
  if (fp8) {
    if (!(k_scale > 0.f) || !isfinite(k_scale) || (has_v && (!(v_scale > 0.f) || !isfinite(v_scale))))
      return fail(PFKV_ERR_INVALID_ARG, "kv_append_fp8: scales must be finite and > 0");
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
  a.slots = slot_mapping;
  a.T = T;
  a.H = H;
  a.D = D;
  a.P = P;
  a.num_pages = num_pages;
  const int64_t n = (int64_t)T * H * (D / 16);
  const int64_t blocks = (n + 255) / 256;
  if (blocks > 0x7FFFFFFF) return fail(PFKV_ERR_UNSUPPORTED, "kv_append: too many tokens");
  dim3 grid((unsigned)blocks, has_v ? 2 : 1);
  if (fp8)
    kv_append_kernel<true><<<grid, 256, 0, stream>>>(a);
  else
    kv_append_kernel<false><<<grid, 256, 0, stream>>>(a);
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
                             num_kv_heads, head_dim, page_size, num_pages, k_scale, v_scale,
                             reinterpret_cast<cudaStream_t>(stream));
}

int pfkv_kv_append_bf16(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                        const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                        int page_size, int64_t num_pages, pfkv_stream_t stream) {
  return pfkv::append_common(false, k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens,
                             num_kv_heads, head_dim, page_size, num_pages, 1.f, 1.f,
                             reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
