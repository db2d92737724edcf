// mla_decode.cu -- MLA absorbed-latent decode over one shared e4m3 latent row
// per token, optionally restricted to a top-k token list.
//
// kLLM article (快手万擎大模型推理成本和性能优化实践), §5.1.1: DSA selects the
// top-k historical tokens that take part in attention and MLA stores a
// compressed per-token latent cKV; §5.1.2: that latent is shared by all heads
// (it cannot be split by head the way GQA KV heads can).  Absorbed reading: the
// whole Dqk = 576-wide row is the key, its first 512 entries are the value.
//
// This translation unit holds the CUDA-core kernel: one CTA per (request,
// 16 heads), 64-token tiles of gathered latent rows in shared memory, online
// softmax per head.  It computes the same function as the tensor-core path and
// is the reference GPU implementation for every supported shape.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "pfkv_internal.h"
#include "pfkv_ptx.cuh"

namespace pfkv {
namespace {

constexpr int kDqk = 576, kDv = 512;
constexpr int kHeadsPerCta = 16;
constexpr int kTok = 64;            // tokens per tile
constexpr int kRowStride = 584;     // bytes per staged row (8-byte aligned, bank spread)
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct MlaArgs {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const uint8_t* ckv;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* topk;
  float* lse;
  int32_t* status;
  int topk_n, B, H, P, max_pages;
  int64_t num_pages;
  float score_scale;  // ckv_scale * softmax_scale * log2(e)
  float out_scale;    // ckv_scale
};

__device__ __forceinline__ float4 e4m3x4_to_f32(uint32_t w) {
  const uint32_t a = e4m3x2_to_f16x2(w & 0xFFFFu), b = e4m3x2_to_f16x2(w >> 16);
  const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&a));
  const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&b));
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}

__global__ void __launch_bounds__(kThreads) mla_decode_cuda_core_kernel(const MlaArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* qs = reinterpret_cast<float*>(smem);                              // [16][576]
  uint8_t* rows = smem + kHeadsPerCta * kDqk * sizeof(float);              // [64][584]
  float* sc = reinterpret_cast<float*>(rows + kTok * kRowStride);          // [16][64]
  int* valid = reinterpret_cast<int*>(sc + kHeadsPerCta * kTok);           // [64]

  const int b = blockIdx.x, h0 = blockIdx.y * kHeadsPerCta;
  const int tid = threadIdx.x;
  const int hh = tid >> 4, sub = tid & 15;

  for (int i = tid; i < kHeadsPerCta * kDqk / 2; i += kThreads) {
    const int h = (2 * i) / kDqk, d = (2 * i) % kDqk;
    const uint32_t v = *reinterpret_cast<const uint32_t*>(
        reinterpret_cast<const uint16_t*>(a.q) + ((int64_t)b * a.H + h0 + h) * kDqk + d);
    qs[h * kDqk + d] = bf16_lo(v);
    qs[h * kDqk + d + 1] = bf16_hi(v);
  }
  int L = a.context_lens[b];
  if (L < 0) L = 0;
  if (L > a.max_pages * a.P) L = a.max_pages * a.P;
  const int n = a.topk ? a.topk_n : L;

  float m = -INFINITY, l = 0.f;
  float o[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) o[j] = 0.f;

  for (int t0 = 0; t0 < n; t0 += kTok) {
    __syncthreads();  // previous tile fully consumed (and q staged on the first pass)
    // ---- gather 64 rows: thread tid copies 8-byte pieces
    for (int r = tid >> 2; r < kTok; r += kThreads >> 2) {
      int tok = -1;
      if (t0 + r < n) tok = a.topk ? a.topk[(int64_t)b * a.topk_n + t0 + r] : t0 + r;
      bool ok = tok >= 0 && tok < L;
      if (a.topk && tok >= L && (tid & 3) == 0) atomicOr(a.status, kErrBadTopk);
      int64_t row = 0;
      if (ok) {
        const int page = a.block_tables[(int64_t)b * a.max_pages + tok / a.P];
        if (page < 0 || page >= a.num_pages) {
          if ((tid & 3) == 0) atomicOr(a.status, kErrBadPage);
          ok = false;
        } else {
          row = (int64_t)page * a.P + tok % a.P;
        }
      }
      if ((tid & 3) == 0) valid[r] = ok;
      const uint2* src = reinterpret_cast<const uint2*>(a.ckv + row * kDqk);
      uint2* dst = reinterpret_cast<uint2*>(rows + r * kRowStride);
      for (int k = tid & 3; k < kDqk / 8; k += 4) dst[k] = ok ? src[k] : make_uint2(0, 0);
    }
    __syncthreads();
    // ---- scores: head hh, tokens sub + 16k
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const float* qh = qs + hh * kDqk;
    for (int w = 0; w < kDqk / 4; ++w) {
      const float4 qv = *reinterpret_cast<const float4*>(qh + 4 * w);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t cw = *reinterpret_cast<const uint32_t*>(rows + (sub + 16 * k) * kRowStride + 4 * w);
        const float4 c = e4m3x4_to_f32(cw);
        acc[k] += qv.x * c.x + qv.y * c.y + qv.z * c.z + qv.w * c.w;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = sub + 16 * k;
      sc[hh * kTok + r] = valid[r] ? acc[k] * a.score_scale : -INFINITY;
    }
    __syncthreads();
    // ---- online softmax for head hh (every thread of the head group redundantly)
    float mx = -INFINITY;
    for (int r = 0; r < kTok; ++r) mx = fmaxf(mx, sc[hh * kTok + r]);
    const float mn = fmaxf(m, mx);
    if (mn == -INFINITY) continue;  // nothing valid yet for this head
    const float al = fast_exp2(m - mn);
    l *= al;
#pragma unroll
    for (int j = 0; j < 32; ++j) o[j] *= al;
    m = mn;
    for (int r = 0; r < kTok; ++r) {
      const float p = fast_exp2(sc[hh * kTok + r] - mn);
      if (p == 0.f) continue;
      l += p;
      const uint8_t* vr = rows + r * kRowStride + sub * 32;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float4 c = e4m3x4_to_f32(*reinterpret_cast<const uint32_t*>(vr + 4 * w));
        o[4 * w] += p * c.x;
        o[4 * w + 1] += p * c.y;
        o[4 * w + 2] += p * c.z;
        o[4 * w + 3] += p * c.w;
      }
    }
  }
  const int64_t head = (int64_t)b * a.H + h0 + hh;
  uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + head * kDv + sub * 32;
  const float inv = l > 0.f ? a.out_scale / l : 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint4 pk;
    pk.x = pack_bf16x2(o[8 * w] * inv, o[8 * w + 1] * inv);
    pk.y = pack_bf16x2(o[8 * w + 2] * inv, o[8 * w + 3] * inv);
    pk.z = pack_bf16x2(o[8 * w + 4] * inv, o[8 * w + 5] * inv);
    pk.w = pack_bf16x2(o[8 * w + 6] * inv, o[8 * w + 7] * inv);
    reinterpret_cast<uint4*>(dst)[w] = pk;
  }
  if (a.lse && sub == 0) a.lse[head] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
}

constexpr size_t kSmemBytes = kHeadsPerCta * kDqk * sizeof(float) + kTok * kRowStride +
                              kHeadsPerCta * kTok * sizeof(float) + kTok * sizeof(int);

}  // namespace
}  // namespace pfkv

extern "C" {

size_t pfkv_mla_decode_workspace_size(int batch, int num_heads, int d_latent, int topk) {
  (void)batch;
  (void)num_heads;
  (void)d_latent;
  (void)topk;
  return 256;  // status word
}

int pfkv_mla_decode_attn(void* out, const void* q, const void* ckv_cache, const int32_t* block_tables,
                         int max_pages_per_seq, const int32_t* context_lens, const int32_t* topk_idx,
                         int topk, int batch, int num_heads, int d_latent, int d_rope, int page_size,
                         int64_t num_pages, float ckv_scale, float softmax_scale, void* workspace,
                         size_t workspace_bytes, float* lse_out, pfkv_stream_t stream) {
  using namespace pfkv;
  clear_error();
  if (batch < 0 || num_heads <= 0 || page_size <= 0 || num_pages <= 0 || max_pages_per_seq <= 0 ||
      (topk_idx && topk <= 0))
    return fail(PFKV_ERR_INVALID_ARG, "mla_decode: bad sizes");
  if (d_latent != kDv || d_rope != kDqk - kDv)
    return fail(PFKV_ERR_UNSUPPORTED, "mla_decode: only d_latent 512 + d_rope 64 supported");
  if (num_heads % kHeadsPerCta != 0 || num_heads > 128)
    return fail(PFKV_ERR_UNSUPPORTED, "mla_decode: num_heads must be a multiple of 16, <= 128");
  if (page_size % 16 != 0)
    return fail(PFKV_ERR_UNSUPPORTED, "mla_decode: page_size must be a multiple of 16");
  if (!isfinite(ckv_scale) || !isfinite(softmax_scale) || !(softmax_scale > 0.f))
    return fail(PFKV_ERR_INVALID_ARG, "mla_decode: scales must be finite");
  if (batch == 0) return PFKV_OK;
  if (!out || !q || !ckv_cache || !block_tables || !context_lens || !workspace)
    return fail(PFKV_ERR_INVALID_ARG, "mla_decode: null pointer");
  if (workspace_bytes < 256) return fail(PFKV_ERR_WORKSPACE, "mla_decode: workspace too small");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(ckv_cache, 16) || !aligned(workspace, 256))
    return fail(PFKV_ERR_INVALID_ARG, "mla_decode: misaligned pointer");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MlaArgs a;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.ckv = static_cast<const uint8_t*>(ckv_cache);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.topk = topk_idx;
  a.lse = lse_out;
  a.status = static_cast<int32_t*>(workspace);
  a.topk_n = topk_idx ? topk : 0;
  a.B = batch;
  a.H = num_heads;
  a.P = page_size;
  a.max_pages = max_pages_per_seq;
  a.num_pages = num_pages;
  a.score_scale = ckv_scale * softmax_scale * kLog2e;
  a.out_scale = ckv_scale;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(mla_decode_cuda_core_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
      return check_cuda("mla_decode set smem attribute");
    attr_set = true;
  }
  if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), s) != cudaSuccess)
    return check_cuda("mla_decode status reset");
  dim3 grid(batch, num_heads / kHeadsPerCta);
  mla_decode_cuda_core_kernel<<<grid, kThreads, kSmemBytes, s>>>(a);
  return check_cuda("mla_decode launch");
}

}  // extern "C"
