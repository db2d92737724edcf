// paged_decode.cu -- GQA/MHA decode attention over a paged e4m3 (or bf16) KV
// cache, dequantised on read, with balanced split-KV and a log-sum-exp merge.
//
// Sources (web pages):
//  * Inference-engine scheduling explainer (推論エンジンの実践), section
//    "PagedAttention の 2 つの原語": KV lives in fixed-size pages and the
//    attention kernel resolves addresses through block_table; section
//    "算力利用率が低いのは表の現象、メモリウォールが根因": decode re-reads the KV
//    from HBM every step and is memory-bound.
//  * Workers AI post (より小さく、高速で、安全に), §1: the FP8 attention kernel
//    converts e4m3 values while reading them.
//  * kLLM article (快手万擎大模型推理成本和性能优化实践), §5.2.2: blockwise
//    attention carries (m, ℓ, O) so that merged blocks equal full attention.
//
// Design (GB300):
//  * Work = 16-token tiles of every (request, KV head), flattened in request-
//    major order.  A persistent grid (SM count x resident CTAs) gives each warp
//    one contiguous run of tiles of equal length (to within one tile), so any
//    mix of context lengths is balanced without host knowledge of the lengths.
//    A run that covers a whole (request, KV head) writes the final output; the
//    others write fp32 (m, ℓ, o) partials that merge_kernel combines.
//  * Each warp is an independent worker with its own ring of kStages shared-
//    memory stages fed by TMA (cp.async.bulk.tensor, 128-byte swizzle): one
//    stage = the K and V slabs of one 16-token tile of one KV head.  The
//    swizzle makes the fragment loads below bank-conflict free.
//  * Scores and P.V run on warp-level tensor-core MMA (m16n8k16, f32 accumulate):
//    S^T[16 tokens x 8 heads] = K_tile . Q^T, then O^T[128 x 8] += V_tile^T . P^T.
//    The e4m3 -> f16 conversion is exact and fused into the fragment build; the
//    K fragment takes 32 contiguous bytes per thread (the head_dim sum is
//    permuted consistently in Q), the V fragment is built with byte permutes.
//    This keeps the CUDA-core work per KV byte small enough for G = 8 heads
//    per KV head at full HBM bandwidth.
//  * Online softmax in the exp2 domain on warp shuffles; P goes to the second
//    MMA through movmatrix (transpose of the accumulator fragment).
#include <cuda_bf16.h>
#include <math.h>

#include "pfkv_internal.h"
#include "pfkv_ptx.cuh"

namespace pfkv {
namespace {

constexpr int kD = 128;
constexpr int kTile = 16;         // tokens per stage = MMA M (scores) / K (P.V)
constexpr int kWarps = 4;         // independent worker warps per CTA
constexpr int kStages = 4;        // TMA ring depth per warp
constexpr int kPartialStride = 132;  // floats per (slot, head): m, l, -, -, o[128]
constexpr int kMaxGrid = 1024;    // bound on persistent CTAs (sizes the workspace)
constexpr int kMaxWarps = kMaxGrid * kWarps;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeArgs {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* lse;
  int32_t* status;
  int64_t* tile_start;  // [B+1] exclusive prefix of Hkv * ceil(L_b / 16)
  int64_t* unit_start;  // [B+1] exclusive prefix of Hkv * chunks_b
  float* partials;      // [capacity][G][kPartialStride]
  int64_t capacity;
  int B, Hq, Hkv, G, P, max_pages;
  int64_t num_pages;
  int chunk_tiles;      // tiles per split unit
  float score_scale;    // k_scale * softmax_scale * log2(e)
  float out_scale;      // v_scale
};

__device__ __forceinline__ int clamp_len(const DecodeArgs& a, int b) {
  int L = a.context_lens[b];
  const int cap = a.max_pages * a.P;
  L = L < 0 ? 0 : L;
  return L > cap ? cap : L;
}

// ----------------------------------------------------------------- plan
// One CTA: exclusive prefix sums of per-request tile and unit counts.
__global__ void __launch_bounds__(1024) plan_kernel(const DecodeArgs a) {
  __shared__ int64_t warp_tiles[32], warp_units[32];
  __shared__ int64_t carry_tiles, carry_units;
  if (threadIdx.x == 0) {
    *a.status = 0;
    carry_tiles = 0;
    carry_units = 0;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int base = 0; base < a.B; base += 1024) {
    const int b = base + threadIdx.x;
    int64_t nt = 0, nu = 0;
    if (b < a.B) {
      const int raw = a.context_lens[b];
      if (raw < 0 || raw > a.max_pages * a.P) atomicOr(a.status, kErrBadContext);
      const int L = clamp_len(a, b);
      const int tiles = (L + kTile - 1) / kTile;
      nt = (int64_t)tiles * a.Hkv;
      nu = (int64_t)((tiles + a.chunk_tiles - 1) / a.chunk_tiles) * a.Hkv;
    }
    // inclusive warp scan
    int64_t st = nt, su = nu;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t xt = __shfl_up_sync(0xFFFFFFFFu, st, o);
      const int64_t xu = __shfl_up_sync(0xFFFFFFFFu, su, o);
      if (lane >= o) {
        st += xt;
        su += xu;
      }
    }
    if (lane == 31) {
      warp_tiles[wid] = st;
      warp_units[wid] = su;
    }
    __syncthreads();
    if (wid == 0) {
      int64_t wt = warp_tiles[lane], wu = warp_units[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t xt = __shfl_up_sync(0xFFFFFFFFu, wt, o);
        const int64_t xu = __shfl_up_sync(0xFFFFFFFFu, wu, o);
        if (lane >= o) {
          wt += xt;
          wu += xu;
        }
      }
      warp_tiles[lane] = wt;
      warp_units[lane] = wu;
    }
    __syncthreads();
    const int64_t pre_t = (wid ? warp_tiles[wid - 1] : 0) + carry_tiles;
    const int64_t pre_u = (wid ? warp_units[wid - 1] : 0) + carry_units;
    if (b < a.B) {
      a.tile_start[b] = pre_t + st - nt;
      a.unit_start[b] = pre_u + su - nu;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      carry_tiles += warp_tiles[31];
      carry_units += warp_units[31];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    a.tile_start[a.B] = carry_tiles;
    a.unit_start[a.B] = carry_units;
  }
}

// ------------------------------------------------------------- work cursor
struct Cursor {
  int b, kvh, tile, ntiles;
};

__device__ __forceinline__ int ntiles_of(const DecodeArgs& a, int b) {
  return (int)((a.tile_start[b + 1] - a.tile_start[b]) / a.Hkv);
}

__device__ void cursor_seek(Cursor& c, const DecodeArgs& a, int64_t f) {
  int lo = 0, hi = a.B;  // tile_start[lo] <= f < tile_start[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.tile_start[mid] <= f)
      lo = mid;
    else
      hi = mid;
  }
  c.b = lo;
  c.ntiles = ntiles_of(a, lo);
  const int64_t rem = f - a.tile_start[lo];
  c.kvh = (int)(rem / c.ntiles);
  c.tile = (int)(rem - (int64_t)c.kvh * c.ntiles);
}

__device__ void cursor_next(Cursor& c, const DecodeArgs& a) {
  if (++c.tile < c.ntiles) return;
  c.tile = 0;
  if (++c.kvh < a.Hkv) return;
  c.kvh = 0;
  do {
    ++c.b;
  } while (c.b < a.B && a.tile_start[c.b + 1] == a.tile_start[c.b]);
  if (c.b < a.B) c.ntiles = ntiles_of(a, c.b);
}

// Owner warp of flattened tile f under the balanced split [w*W/N, (w+1)*W/N).
__device__ __forceinline__ int64_t owner_of(int64_t f, int64_t W, int64_t N) {
  return ((f + 1) * N - 1) / W;
}

// 128-byte-swizzled offset of 16-byte chunk c of row r inside a [rows][128 B]
// box written by TMA with CU_TENSOR_MAP_SWIZZLE_128B (1024-byte aligned).
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

template <bool kBf16>
struct Geometry {
  static constexpr int kKBytes = kBf16 ? 4096 : 2048;  // one 16-token K slab
  static constexpr int kStageBytes = 2 * kKBytes;       // K + V
  static constexpr int kWarpBytes = kStages * kStageBytes;
  static constexpr int kSmemBytes = kWarps * kWarpBytes + 1024;  // + alignment slack
};

// --------------------------------------------------------------- main kernel
template <bool kBf16, int NT>
__global__ void __launch_bounds__(kWarps * 32)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecodeArgs a) {
  using Geo = Geometry<kBf16>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kWarps][kStages];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t wbase = smem_base + warp * Geo::kWarpBytes;
  uint32_t bar[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) bar[s] = smem_u32(&bars[warp][s]);

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(bar[s], 1);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncwarp();

  const int64_t N = (int64_t)gridDim.x * kWarps;
  const int64_t w = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t W = a.tile_start[a.B];
  const int64_t f_begin = w * W / N, f_end = (w + 1) * W / N;
  if (f_begin >= f_end) return;

  // --- producer: all lanes track the cursor, lane 0 issues.
  Cursor pc;
  cursor_seek(pc, a, f_begin);
  int64_t f_issue = f_begin;
  auto issue = [&](int stage) {
    if (lane == 0) {
      const int tok0 = pc.tile * kTile;
      const int lp = tok0 / a.P;
      int page = a.block_tables[(int64_t)pc.b * a.max_pages + lp];
      if (page < 0 || (int64_t)page >= a.num_pages) {
        atomicOr(a.status, kErrBadPage);
        page = -1;  // the TMA box lands outside the tensor and reads zeros
      }
      const int row = (page * a.Hkv + pc.kvh) * a.P + (tok0 - lp * a.P);
      const uint32_t dst = wbase + stage * Geo::kStageBytes;
      mbar_arrive_expect_tx(bar[stage], Geo::kStageBytes);
      if constexpr (kBf16) {
        tma_load_3d(dst, &tmK, 0, 0, row, bar[stage]);
        tma_load_3d(dst + 2048, &tmK, 0, 1, row, bar[stage]);
        tma_load_3d(dst + Geo::kKBytes, &tmV, 0, 0, row, bar[stage]);
        tma_load_3d(dst + Geo::kKBytes + 2048, &tmV, 0, 1, row, bar[stage]);
      } else {
        tma_load_2d(dst, &tmK, 0, row, bar[stage]);
        tma_load_2d(dst + Geo::kKBytes, &tmV, 0, row, bar[stage]);
      }
    }
    cursor_next(pc, a);
    ++f_issue;
  };
#pragma unroll
  for (int s = 0; s < kStages; ++s)
    if (f_issue < f_end) issue(s);

  // --- consumer state
  Cursor cc;
  cursor_seek(cc, a, f_begin);
  float m[NT][2], l[NT][2], o[NT][8][4];
  uint32_t qf[NT][8][2];
  int L = 0;
  int64_t seg_begin = f_begin;
  bool timed_out = false;

  auto flush = [&](int64_t f_stop) {
    // f_stop: first flattened tile after this segment
    const int b = cc.b, kvh = cc.kvh;  // cursor still on the segment's last tile
    const int ntiles = cc.ntiles;
    const int chunk = cc.tile / a.chunk_tiles;
    const int64_t ts = a.tile_start[b];
    const int64_t s_u = ts + (int64_t)kvh * ntiles + (int64_t)chunk * a.chunk_tiles;
    int64_t e_u = s_u + a.chunk_tiles;
    const int64_t e_req = ts + (int64_t)(kvh + 1) * ntiles;
    if (e_u > e_req) e_u = e_req;
    const int nchunks = (int)((a.unit_start[b + 1] - a.unit_start[b]) / a.Hkv);
    const bool final = (nchunks == 1) && seg_begin == s_u && f_stop == e_u;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = l[j][e];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
        l[j][e] = v;
      }
    const int64_t u = a.unit_start[b] + (int64_t)kvh * nchunks + chunk;
    const int64_t slot = w + u;
    if (!final && slot >= a.capacity) {
      if (lane == 0) atomicOr(a.status, kErrWorkspace);
      return;
    }
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hl = 8 * j + 2 * t + e;
        if (hl >= a.G) continue;
        const int64_t head = (int64_t)b * a.Hq + (int64_t)kvh * a.G + hl;
        // this thread's 16 head_dim values, in two runs of 8 (bf16 cache) or one of 16 (e4m3)
        float vals[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          vals[2 * i] = o[j][i][e];
          vals[2 * i + 1] = o[j][i][2 + e];
        }
        if (final) {
          const float inv = a.out_scale / l[j][e];
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(vals[2 * i] * inv, vals[2 * i + 1] * inv);
          uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + head * kD;
          if constexpr (kBf16) {
            *reinterpret_cast<uint4*>(dst + 8 * g) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(dst + 64 + 8 * g) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          } else {
            *reinterpret_cast<uint4*>(dst + 16 * g) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(dst + 16 * g + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
          if (a.lse && g == 0) a.lse[head] = (m[j][e] + __log2f(l[j][e])) * kLn2;
        } else {
          float* dst = a.partials + (slot * a.G + hl) * kPartialStride;
          if (g == 0) {
            dst[0] = m[j][e];
            dst[1] = l[j][e];
          }
          float4* o4 = reinterpret_cast<float4*>(dst + 4);
          if constexpr (kBf16) {
            o4[2 * g] = make_float4(vals[0], vals[1], vals[2], vals[3]);
            o4[2 * g + 1] = make_float4(vals[4], vals[5], vals[6], vals[7]);
            o4[16 + 2 * g] = make_float4(vals[8], vals[9], vals[10], vals[11]);
            o4[16 + 2 * g + 1] = make_float4(vals[12], vals[13], vals[14], vals[15]);
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              o4[4 * g + k] = make_float4(vals[4 * k], vals[4 * k + 1], vals[4 * k + 2], vals[4 * k + 3]);
          }
        }
      }
  };

  auto start_unit = [&]() {
    L = clamp_len(a, cc.b);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      m[j][0] = m[j][1] = -INFINITY;
      l[j][0] = l[j][1] = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[j][i][0] = o[j][i][1] = o[j][i][2] = o[j][i][3] = 0.f;
      const int hl = 8 * j + g;
      uint4 r[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                    make_uint4(0, 0, 0, 0)};
      if (hl < a.G) {
        const uint4* qp = reinterpret_cast<const uint4*>(
            a.q + ((int64_t)cc.b * a.Hq + (int64_t)cc.kvh * a.G + hl) * kD);
        if constexpr (kBf16) {
          // head_dim values 16t..16t+15 of each 64-wide half
          r[0] = qp[2 * t];
          r[1] = qp[2 * t + 1];
          r[2] = qp[8 + 2 * t];
          r[3] = qp[8 + 2 * t + 1];
        } else {
          // head_dim values 32t..32t+31
#pragma unroll
          for (int k = 0; k < 4; ++k) r[k] = qp[4 * t + k];
        }
      }
      const uint32_t wd[16] = {r[0].x, r[0].y, r[0].z, r[0].w, r[1].x, r[1].y, r[1].z, r[1].w,
                               r[2].x, r[2].y, r[2].z, r[2].w, r[3].x, r[3].y, r[3].z, r[3].w};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        if constexpr (kBf16) {
          qf[j][ks][0] = wd[2 * ks];
          qf[j][ks][1] = wd[2 * ks + 1];
        } else {
          qf[j][ks][0] = pack_f16x2(bf16_lo(wd[2 * ks]), bf16_hi(wd[2 * ks]));
          qf[j][ks][1] = pack_f16x2(bf16_lo(wd[2 * ks + 1]), bf16_hi(wd[2 * ks + 1]));
        }
      }
    }
  };

  int stage = 0;
  uint32_t phase = 0;
  for (int64_t f = f_begin; f < f_end; ++f) {
    if (f == f_begin || cc.tile % a.chunk_tiles == 0) {
      if (f != f_begin) {
        // the cursor has moved on: flush used the previous tile's identity
      }
      start_unit();
      seg_begin = f;
    }
    if (!mbar_wait(bar[stage], phase)) {
      timed_out = true;
      break;
    }
    const uint32_t kb = wbase + stage * Geo::kStageBytes;
    const uint32_t vb = kb + Geo::kKBytes;
    const int tok0 = cc.tile * kTile;

    // ---------------- S^T = K . Q^T  (rows: tokens, cols: heads)
    float s[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
    if constexpr (kBf16) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint32_t hb = kb + h2 * 2048;
        const uint4 x0 = lds128(hb + swz(g, 2 * t)), x1 = lds128(hb + swz(g, 2 * t + 1));
        const uint4 y0 = lds128(hb + swz(g + 8, 2 * t)), y1 = lds128(hb + swz(g + 8, 2 * t + 1));
        const uint32_t xr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const uint32_t yr[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int ks = 4 * h2 + jj;
#pragma unroll
          for (int j = 0; j < NT; ++j)
            mma_bf16(s[j], xr[2 * jj], yr[2 * jj], xr[2 * jj + 1], yr[2 * jj + 1], qf[j][ks][0],
                     qf[j][ks][1]);
        }
      }
    } else {
      const uint4 x0 = lds128(kb + swz(g, 2 * t)), x1 = lds128(kb + swz(g, 2 * t + 1));
      const uint4 y0 = lds128(kb + swz(g + 8, 2 * t)), y1 = lds128(kb + swz(g + 8, 2 * t + 1));
      const uint32_t xr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t yr[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t a0 = e4m3x2_to_f16x2(xr[ks] & 0xFFFFu);
        const uint32_t a1 = e4m3x2_to_f16x2(yr[ks] & 0xFFFFu);
        const uint32_t a2 = e4m3x2_to_f16x2(xr[ks] >> 16);
        const uint32_t a3 = e4m3x2_to_f16x2(yr[ks] >> 16);
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_f16(s[j], a0, a1, a2, a3, qf[j][ks][0], qf[j][ks][1]);
      }
    }

    // ---------------- masking + online softmax (exp2 domain)
    const bool va = tok0 + g < L, vb8 = tok0 + g + 8 < L;
    uint32_t pb[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float s0 = va ? s[j][0] * a.score_scale : -INFINITY;
      const float s1 = va ? s[j][1] * a.score_scale : -INFINITY;
      const float s2 = vb8 ? s[j][2] * a.score_scale : -INFINITY;
      const float s3 = vb8 ? s[j][3] * a.score_scale : -INFINITY;
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
      }
      const float mn0 = fmaxf(m[j][0], mx0), mn1 = fmaxf(m[j][1], mx1);
      const float al0 = fast_exp2(m[j][0] - mn0), al1 = fast_exp2(m[j][1] - mn1);
      const float p0 = fast_exp2(s0 - mn0), p1 = fast_exp2(s1 - mn1);
      const float p2 = fast_exp2(s2 - mn0), p3 = fast_exp2(s3 - mn1);
      l[j][0] = l[j][0] * al0 + (p0 + p2);
      l[j][1] = l[j][1] * al1 + (p1 + p3);
      m[j][0] = mn0;
      m[j][1] = mn1;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        o[j][i][0] *= al0;
        o[j][i][1] *= al1;
        o[j][i][2] *= al0;
        o[j][i][3] *= al1;
      }
      if constexpr (kBf16) {
        pb[j][0] = movmatrix_trans(pack_bf16x2(p0, p1));
        pb[j][1] = movmatrix_trans(pack_bf16x2(p2, p3));
      } else {
        pb[j][0] = movmatrix_trans(pack_f16x2(p0, p1));
        pb[j][1] = movmatrix_trans(pack_f16x2(p2, p3));
      }
    }

    // ---------------- O^T += V^T . P^T  (rows: head_dim, cols: heads)
    const bool partial = tok0 + kTile > L;
    const bool v0ok = tok0 + 2 * t < L, v1ok = tok0 + 2 * t + 1 < L;
    const bool v2ok = tok0 + 2 * t + 8 < L, v3ok = tok0 + 2 * t + 9 < L;
    if constexpr (kBf16) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint32_t hb = vb + h2 * 2048;
        uint4 r0 = lds128(hb + swz(2 * t, g)), r1 = lds128(hb + swz(2 * t + 1, g));
        uint4 r2 = lds128(hb + swz(2 * t + 8, g)), r3 = lds128(hb + swz(2 * t + 9, g));
        if (partial) {
          const uint4 z = make_uint4(0, 0, 0, 0);
          if (!v0ok) r0 = z;
          if (!v1ok) r1 = z;
          if (!v2ok) r2 = z;
          if (!v3ok) r3 = z;
        }
        const uint32_t R0[4] = {r0.x, r0.y, r0.z, r0.w}, R1[4] = {r1.x, r1.y, r1.z, r1.w};
        const uint32_t R2[4] = {r2.x, r2.y, r2.z, r2.w}, R3[4] = {r3.x, r3.y, r3.z, r3.w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int i = 4 * h2 + jj;
          const uint32_t A0 = prmt(R0[jj], R1[jj], 0x5410), A1 = prmt(R0[jj], R1[jj], 0x7632);
          const uint32_t A2 = prmt(R2[jj], R3[jj], 0x5410), A3 = prmt(R2[jj], R3[jj], 0x7632);
#pragma unroll
          for (int j = 0; j < NT; ++j) mma_bf16(o[j][i], A0, A1, A2, A3, pb[j][0], pb[j][1]);
        }
      }
    } else {
      uint4 r0 = lds128(vb + swz(2 * t, g)), r1 = lds128(vb + swz(2 * t + 1, g));
      uint4 r2 = lds128(vb + swz(2 * t + 8, g)), r3 = lds128(vb + swz(2 * t + 9, g));
      if (partial) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        if (!v0ok) r0 = z;
        if (!v1ok) r1 = z;
        if (!v2ok) r2 = z;
        if (!v3ok) r3 = z;
      }
      const uint32_t R0[4] = {r0.x, r0.y, r0.z, r0.w}, R1[4] = {r1.x, r1.y, r1.z, r1.w};
      const uint32_t R2[4] = {r2.x, r2.y, r2.z, r2.w}, R3[4] = {r3.x, r3.y, r3.z, r3.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
        const uint32_t x01 = prmt(R0[i >> 1], R1[i >> 1], sel);
        const uint32_t x23 = prmt(R2[i >> 1], R3[i >> 1], sel);
        const uint32_t A0 = e4m3x2_to_f16x2(x01 & 0xFFFFu), A1 = e4m3x2_to_f16x2(x01 >> 16);
        const uint32_t A2 = e4m3x2_to_f16x2(x23 & 0xFFFFu), A3 = e4m3x2_to_f16x2(x23 >> 16);
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_f16(o[j][i], A0, A1, A2, A3, pb[j][0], pb[j][1]);
      }
    }

    // ---------------- refill this stage with the tile kStages ahead
    __syncwarp();
    if (f_issue < f_end) {
      if (lane == 0) fence_proxy_async_smem();
      issue(stage);
    }
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }

    // ---------------- end of a unit segment?
    const int64_t fn = f + 1;
    bool boundary = (fn == f_end);
    if (!boundary) {
      const int nt = cc.tile + 1;
      boundary = (nt == cc.ntiles) || (nt % a.chunk_tiles == 0);
    }
    if (boundary) flush(fn);
    cursor_next(cc, a);
  }

  if (timed_out) {
    if (lane == 0) atomicOr(a.status, kErrWaitTimeout);
    // let every copy still in flight land before the CTA's memory is released
    for (int s = 0; s < kStages; ++s) (void)mbar_wait(bar[s], 0), (void)mbar_wait(bar[s], 1);
  }
}

// -------------------------------------------------------------- merge kernel
// One CTA per (request, KV head); G warps, one per query head, each lane owns
// four head_dim values.  Combines the fp32 partials of every segment with the
// log-sum-exp rule: M = max m_k, out = sum 2^{m_k-M} o_k / sum 2^{m_k-M} l_k.
__global__ void __launch_bounds__(512) merge_kernel(const DecodeArgs a, int64_t N) {
  const int b = blockIdx.x / a.Hkv, kvh = blockIdx.x % a.Hkv;
  const int hl = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (hl >= a.G) return;
  const int64_t head = (int64_t)b * a.Hq + (int64_t)kvh * a.G + hl;
  uint2* out2 = reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + head * kD) + lane;
  const int ntiles = ntiles_of(a, b);
  if (ntiles == 0) {
    *out2 = make_uint2(0, 0);
    if (a.lse && lane == 0) a.lse[head] = -INFINITY;
    return;
  }
  const int64_t W = a.tile_start[a.B];
  const int nchunks = (int)((a.unit_start[b + 1] - a.unit_start[b]) / a.Hkv);
  const int64_t ts = a.tile_start[b] + (int64_t)kvh * ntiles;
  const int64_t u0 = a.unit_start[b] + (int64_t)kvh * nchunks;
  if (nchunks == 1 && owner_of(ts, W, N) == owner_of(ts + ntiles - 1, W, N)) return;  // direct

  float M = -INFINITY;
  for (int c = 0; c < nchunks; ++c) {
    const int64_t s_u = ts + (int64_t)c * a.chunk_tiles;
    const int64_t e_u = min(s_u + a.chunk_tiles, ts + ntiles);
    const int64_t w1 = owner_of(e_u - 1, W, N);
    for (int64_t w = owner_of(s_u, W, N); w <= w1; ++w) {
      if (w * W / N == (w + 1) * W / N) continue;  // a warp with no tiles wrote nothing
      const int64_t slot = w + u0 + c;
      if (slot < a.capacity) M = fmaxf(M, a.partials[(slot * a.G + hl) * kPartialStride]);
    }
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int c = 0; c < nchunks; ++c) {
    const int64_t s_u = ts + (int64_t)c * a.chunk_tiles;
    const int64_t e_u = min(s_u + a.chunk_tiles, ts + ntiles);
    const int64_t w1 = owner_of(e_u - 1, W, N);
    for (int64_t w = owner_of(s_u, W, N); w <= w1; ++w) {
      if (w * W / N == (w + 1) * W / N) continue;
      const int64_t slot = w + u0 + c;
      if (slot >= a.capacity) continue;
      const float* p = a.partials + (slot * a.G + hl) * kPartialStride;
      const float wt = fast_exp2(p[0] - M);
      den += wt * p[1];
      const float4 v = reinterpret_cast<const float4*>(p + 4)[lane];
      acc.x += wt * v.x;
      acc.y += wt * v.y;
      acc.z += wt * v.z;
      acc.w += wt * v.w;
    }
  }
  const float inv = a.out_scale / den;
  *out2 = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (a.lse && lane == 0) a.lse[head] = (M + __log2f(den)) * kLn2;
}

// ------------------------------------------------------------------- host
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t tile_off, unit_off, part_off;
};

WsLayout ws_layout(int B) {
  WsLayout L;
  L.tile_off = 256;
  L.unit_off = align_up(L.tile_off + sizeof(int64_t) * (size_t)(B + 1), 256);
  L.part_off = align_up(L.unit_off + sizeof(int64_t) * (size_t)(B + 1), 256);
  return L;
}

template <bool kBf16, int NT>
int launch_decode(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeArgs& a,
                  cudaStream_t stream) {
  using Geo = Geometry<kBf16>;
  auto kern = paged_decode_kernel<kBf16, NT>;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Geo::kSmemBytes) !=
        cudaSuccess)
      return check_cuda("paged_decode set smem attribute");
    attr_set = true;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, Geo::kSmemBytes) !=
      cudaSuccess)
    return check_cuda("paged_decode occupancy");
  if (per_sm < 1) per_sm = 1;
  int grid = device_sm_count() * per_sm;
  if (grid < 1) grid = 1;
  if (grid > kMaxGrid) grid = kMaxGrid;
  plan_kernel<<<1, 1024, 0, stream>>>(a);
  kern<<<grid, kWarps * 32, Geo::kSmemBytes, stream>>>(tmK, tmV, a);
  merge_kernel<<<a.B * a.Hkv, a.G * 32, 0, stream>>>(a, (int64_t)grid * kWarps);
  return check_cuda("paged_decode launch");
}

}  // namespace
}  // namespace pfkv

extern "C" {

size_t pfkv_paged_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                        int kv_split_tokens, int64_t max_total_chunks) {
  (void)head_dim;
  if (batch < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads) return 0;
  const int G = num_q_heads / num_kv_heads;
  int64_t units = batch;
  if (kv_split_tokens > 0 && max_total_chunks > units) units = max_total_chunks;
  const pfkv::WsLayout L = pfkv::ws_layout(batch);
  const int64_t slots = pfkv::kMaxWarps + (int64_t)num_kv_heads * units;
  return L.part_off + (size_t)slots * G * pfkv::kPartialStride * sizeof(float);
}

int pfkv_paged_decode_attn(void* out, const void* q, const void* k_cache, const void* v_cache,
                           pfkv_cache_dtype cache_dtype, const int32_t* block_tables,
                           int max_pages_per_seq, const int32_t* context_lens, int batch,
                           int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                           int64_t num_pages, float k_scale, float v_scale, float softmax_scale,
                           int kv_split_tokens, void* workspace, size_t workspace_bytes,
                           float* lse_out, pfkv_stream_t stream) {
  using namespace pfkv;
  clear_error();
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || page_size <= 0 || num_pages <= 0 ||
      max_pages_per_seq <= 0)
    return fail(PFKV_ERR_INVALID_ARG, "paged_decode: bad sizes");
  if (num_q_heads % num_kv_heads != 0)
    return fail(PFKV_ERR_INVALID_ARG, "paged_decode: num_q_heads %% num_kv_heads != 0");
  const int G = num_q_heads / num_kv_heads;
  if (G > 16) return fail(PFKV_ERR_UNSUPPORTED, "paged_decode: group size %d > 16", G);
  if (head_dim != kD) return fail(PFKV_ERR_UNSUPPORTED, "paged_decode: head_dim %d != 128", head_dim);
  if (page_size % kTile != 0)
    return fail(PFKV_ERR_UNSUPPORTED, "paged_decode: page_size %d not a multiple of 16", page_size);
  if (kv_split_tokens < 0 || kv_split_tokens % kTile != 0)
    return fail(PFKV_ERR_INVALID_ARG, "paged_decode: kv_split_tokens must be a multiple of 16");
  if (cache_dtype != PFKV_CACHE_FP8_E4M3 && cache_dtype != PFKV_CACHE_BF16)
    return fail(PFKV_ERR_INVALID_ARG, "paged_decode: unknown cache dtype");
  if ((int64_t)num_pages * num_kv_heads * page_size >= (int64_t)1 << 31)
    return fail(PFKV_ERR_UNSUPPORTED, "paged_decode: cache has 2^31 or more token rows");
  if ((int64_t)max_pages_per_seq * page_size >= (int64_t)1 << 30)
    return fail(PFKV_ERR_UNSUPPORTED, "paged_decode: block table too long");
  if (!(softmax_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale) || !isfinite(softmax_scale))
    return fail(PFKV_ERR_INVALID_ARG, "paged_decode: scales must be finite");
  if (batch == 0) return PFKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace)
    return fail(PFKV_ERR_INVALID_ARG, "paged_decode: null pointer");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(workspace, 256) || !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
      (lse_out && !aligned(lse_out, 4)))
    return fail(PFKV_ERR_INVALID_ARG, "paged_decode: misaligned pointer");
  const WsLayout L = ws_layout(batch);
  const size_t per_slot = (size_t)G * kPartialStride * sizeof(float);
  if (workspace_bytes < L.part_off + per_slot * ((size_t)kMaxWarps + (size_t)num_kv_heads * batch))
    return fail(PFKV_ERR_WORKSPACE, "paged_decode: workspace of %zu bytes is too small",
                workspace_bytes);

  DecodeArgs a;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.lse = lse_out;
  a.status = reinterpret_cast<int32_t*>(ws);
  a.tile_start = reinterpret_cast<int64_t*>(ws + L.tile_off);
  a.unit_start = reinterpret_cast<int64_t*>(ws + L.unit_off);
  a.partials = reinterpret_cast<float*>(ws + L.part_off);
  a.capacity = (int64_t)((workspace_bytes - L.part_off) / per_slot);
  a.B = batch;
  a.Hq = num_q_heads;
  a.Hkv = num_kv_heads;
  a.G = G;
  a.P = page_size;
  a.max_pages = max_pages_per_seq;
  a.num_pages = num_pages;
  a.chunk_tiles = kv_split_tokens > 0 ? kv_split_tokens / kTile : (1 << 30);
  a.score_scale = k_scale * softmax_scale * kLog2e;
  a.out_scale = v_scale;

  const bool bf16 = cache_dtype == PFKV_CACHE_BF16;
  const cuuint64_t rows = (cuuint64_t)num_pages * num_kv_heads * page_size;
  CUtensorMap tmK, tmV;
  int rc;
  if (bf16) {
    const cuuint64_t dims[3] = {64, 2, rows};
    const cuuint64_t strides[2] = {128, 256};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kTile};
    rc = encode_tensor_map(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k_cache), dims,
                           strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc == PFKV_OK)
      rc = encode_tensor_map(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v_cache),
                             dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const cuuint64_t dims[2] = {128, rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, (cuuint32_t)kTile};
    rc = encode_tensor_map(&tmK, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(k_cache), dims,
                           strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc == PFKV_OK)
      rc = encode_tensor_map(&tmV, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(v_cache), dims,
                             strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (rc != PFKV_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (bf16)
    return G <= 8 ? launch_decode<true, 1>(tmK, tmV, a, s) : launch_decode<true, 2>(tmK, tmV, a, s);
  return G <= 8 ? launch_decode<false, 1>(tmK, tmV, a, s) : launch_decode<false, 2>(tmK, tmV, a, s);
}

}  // extern "C"
