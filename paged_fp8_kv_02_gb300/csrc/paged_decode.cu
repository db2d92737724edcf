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
//    others write fp32 (m, ℓ, o) partials that a merge kernel combines (one
//    warp per query head for calls without explicit chunks).
//  * Each warp is an independent worker with its own ring of kStages shared-
//    memory stages fed by TMA (cp.async.bulk.tensor, 128-byte swizzle): one
//    stage = the K and V slabs of one 16-token tile of one KV head.  The
//    swizzle makes the fragment loads below bank-conflict free.
//  * Scores and P.V run on warp-level tensor-core MMA with f32 accumulation:
//    S^T[16 tokens x 8 heads] = K_tile . Q^T, then O^T[128 x 8] += V_tile^T . P^T.
//    e4m3 cache: the scores are m16n8k32 e4m3 products straight on the K bytes
//    in shared memory (each thread's K fragment is 32 contiguous bytes of a
//    row; the head_dim sum is permuted the same way in Q) against Q split per
//    head into two exact e4m3 parts after a power-of-two scale; the per-token-
//    scale variant widens K to f16 instead (m16n8k16).  V widens to f16
//    (exact) inside the fragment build, with byte permutes.  bf16 cache: bf16
//    products for both.  This keeps the CUDA-core work per KV byte small
//    enough for G = 8 heads per KV head at full HBM bandwidth.
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
constexpr int kStages = 3;        // TMA ring depth per warp
// floats per (slot, head): m, l, -, -, o[128], padded to five whole 128-byte
// lines so that the merge can drop a state's lines from L2 once it is folded
constexpr int kPartialStride = 160;
static_assert(kPartialStride * sizeof(float) % 128 == 0, "partial states must be whole L2 lines");
constexpr int kMaxGrid = 1024;    // bound on persistent CTAs (sizes the workspace)
constexpr int kMaxWarps = kMaxGrid * kWarps;
constexpr float kLog2e = 1.4426950408889634f;
// Where the K/V scales come from: host scalars in DecodeArgs, one device scale
// per work unit (per tensor or per KV head), or one per token row.
enum : int { kSclHost = 0, kSclUnit = 1, kSclToken = 2 };
constexpr int kScaleStageBytes = 128;  // per-token mode: 16 K + 16 V fp32 scales per stage
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
  int64_t capacity;     // partial slots (and the bound on units)
  int64_t nwarps;       // warps of the tile kernel's grid
  int B, Hq, Hkv, G, P, max_pages;
  int64_t num_pages;
  int chunk_tiles;      // tiles per split unit
  float score_scale;    // k_scale * softmax_scale * log2(e)
  float out_scale;      // v_scale
  const float* k_scales;   // device scales (unit or token modes)
  const float* v_scales;
  int scale_head_stride;   // unit mode: 1 = one scale per KV head, 0 = one for all
  float logit_scale;       // softmax_scale * log2(e)
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
  grid_launch_dependents();  // the tile kernel may start its prologue now
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
    if (carry_units > a.capacity) atomicOr(a.status, kErrWorkspace);
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

template <bool kBf16, int kScl = kSclHost>
struct Geometry {
  static constexpr int kKBytes = kBf16 ? 4096 : 2048;  // one 16-token K slab
  static constexpr int kStageBytes = 2 * kKBytes;       // K + V
  static constexpr int kWarpBytes = kStages * kStageBytes;
  // per-token scales sit after all warps' tiles (which keep their 1024-byte alignment)
  static constexpr int kScaleWarpBytes = kScl == kSclToken ? kStages * kScaleStageBytes : 0;
  static constexpr int kSmemBytes = kWarps * (kWarpBytes + kScaleWarpBytes) + 1024;  // + alignment slack
};

// --------------------------------------------------------------- main kernel
// Lazy softmax rescale: the running reference max of a head is only raised when
// a score exceeds it by more than kRescaleLog2 (log2 units); in between, p =
// 2^(s - ref) stays <= 2^kRescaleLog2, which f16/bf16 P and the fp32
// accumulators carry with unchanged relative precision.  The reference is a
// pure re-parametrisation: (ref, l, o) describe the same state as the exact
// running maximum would.
constexpr float kRescaleLog2 = 8.f;

template <bool kBf16, int NT, int kScl>
__global__ void __launch_bounds__(kWarps * 32, NT == 1 ? 4 : 2)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecodeArgs a) {
  static_assert(!kBf16 || kScl == kSclHost, "device scales are for the e4m3 cache");
  using Geo = Geometry<kBf16, kScl>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kWarps][kStages];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t wbase = smem_base + warp * Geo::kWarpBytes;
  uint8_t* const wptr = smem_raw + (smem_base - smem_u32(smem_raw)) + warp * Geo::kWarpBytes;
  // per-token mode: this warp's kStages x (16 K + 16 V) fp32 scales
  const uint32_t sbase = smem_base + kWarps * Geo::kWarpBytes + warp * Geo::kScaleWarpBytes;
  float* const sptr = reinterpret_cast<float*>(wptr + (kWarps - warp) * Geo::kWarpBytes +
                                               warp * Geo::kScaleWarpBytes);
  const uint32_t bar0 = smem_u32(&bars[warp][0]);  // stage s: bar0 + 8 s

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncwarp();
  grid_launch_dependents();  // the merge kernel may be scheduled as CTAs retire
  grid_dependency_wait();    // the plan's prefix sums are complete and visible

  const int64_t N = (int64_t)gridDim.x * kWarps;
  const int64_t w = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t W = a.tile_start[a.B];
  const int64_t f_begin = w * W / N, f_end = (w + 1) * W / N;
  if (f_begin >= f_end) return;

  // --- producer: all lanes track the cursor, lane 0 issues.  The block-table
  // entry of the next tile to issue is loaded one issue ahead, so the TMA issue
  // never waits on a dependent global load.
  Cursor pc;
  cursor_seek(pc, a, f_begin);
  int64_t f_issue = f_begin;
  int next_page = 0;
  auto load_page = [&]() {
    if (lane == 0 && f_issue < f_end)
      next_page = __ldg(a.block_tables + (int64_t)pc.b * a.max_pages + (pc.tile * kTile) / a.P);
  };
  load_page();
  const uint64_t kv_policy = l2_evict_first_policy();  // K/V is read once
  auto issue = [&](int stage) {
    if (lane == 0) {
      const int tok0 = pc.tile * kTile;
      int page = next_page;
      if (page < 0 || (int64_t)page >= a.num_pages) {
        atomicOr(a.status, kErrBadPage);
        page = -1;  // the TMA box lands outside the tensor and reads zeros
      }
      const int row = (page * a.Hkv + pc.kvh) * a.P + tok0 % a.P;
      const uint32_t dst = wbase + stage * Geo::kStageBytes;
      const uint32_t bar = bar0 + 8 * stage;
      uint32_t tx = Geo::kStageBytes;
      if constexpr (kScl == kSclToken) {
        if (page >= 0) {
          tx += kScaleStageBytes;
        } else {  // a row outside the pool: zero scales beside its zero codes
          float4* z = reinterpret_cast<float4*>(sptr + stage * (kScaleStageBytes / 4));
#pragma unroll
          for (int i = 0; i < kScaleStageBytes / 16; ++i) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      mbar_arrive_expect_tx(bar, tx);
      if constexpr (kScl == kSclToken) {
        if (page >= 0) {
          const uint32_t sdst = sbase + stage * kScaleStageBytes;
          bulk_load(sdst, a.k_scales + row, 64, bar);
          bulk_load(sdst + 64, a.v_scales + row, 64, bar);
        }
      }
      if constexpr (kBf16) {
        tma_load_3d_hint(dst, &tmK, 0, 0, row, bar, kv_policy);
        tma_load_3d_hint(dst + 2048, &tmK, 0, 1, row, bar, kv_policy);
        tma_load_3d_hint(dst + Geo::kKBytes, &tmV, 0, 0, row, bar, kv_policy);
        tma_load_3d_hint(dst + Geo::kKBytes + 2048, &tmV, 0, 1, row, bar, kv_policy);
      } else {
        tma_load_2d_hint(dst, &tmK, 0, row, bar, kv_policy);
        tma_load_2d_hint(dst + Geo::kKBytes, &tmV, 0, row, bar, kv_policy);
      }
    }
    cursor_next(pc, a);
    ++f_issue;
    load_page();
  };
#pragma unroll
  for (int s = 0; s < kStages; ++s)
    if (f_issue < f_end) issue(s);

  // --- consumer state
  Cursor cc;
  cursor_seek(cc, a, f_begin);
  float mref[NT][2];   // reference max per head (log2 domain, scaled scores)
  float rthr[NT][2];   // raw-score threshold that forces a rescale
  float l[NT][2], o[NT][8][4];
  uint32_t qf[NT][8][2];
  int L = 0;
  int chunk_left = 0;  // tiles left in the current unit, including the current one
  int64_t seg_begin = f_begin;
  float sc = a.score_scale;  // unit mode: set per unit from the device K scale
  // e4m3 cache: 1 / the power-of-two Q scale, per head of the score columns
  // 2t and 2t + 1 of each head tile (per unit for per-token scales)
  float qinv[NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j) qinv[j][0] = qinv[j][1] = 1.f;
  float unit_vs = 1.f;       // unit mode: the unit's V scale
  float vref = 0.f, vinv = 0.f;  // token mode: largest V scale of the unit so far, 1 / it

  auto flush = [&](int64_t f_stop) {
    // f_stop: first flattened tile after this segment; cc is on its last tile
    const int b = cc.b, kvh = cc.kvh;
    const int ntiles = cc.ntiles;
    const int chunk = cc.tile / a.chunk_tiles;
    const int64_t ts = a.tile_start[b];
    const int64_t s_u = ts + (int64_t)kvh * ntiles + (int64_t)chunk * a.chunk_tiles;
    int64_t e_u = s_u + a.chunk_tiles;
    const int64_t e_req = ts + (int64_t)(kvh + 1) * ntiles;
    if (e_u > e_req) e_u = e_req;
    const int nchunks = (int)((a.unit_start[b + 1] - a.unit_start[b]) / a.Hkv);
    const bool final = (nchunks == 1) && seg_begin == s_u && f_stop == e_u;
    // factor from accumulator units to dequantised V units
    const float vmul = kScl == kSclUnit ? unit_vs : (kScl == kSclToken ? vref : 1.f);
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
        if constexpr (kScl != kSclHost) {
#pragma unroll
          for (int i = 0; i < 16; ++i) vals[i] *= vmul;
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
          if (a.lse && g == 0) a.lse[head] = (mref[j][e] + __log2f(l[j][e])) * kLn2;
        } else {
          float* dst = a.partials + (slot * a.G + hl) * kPartialStride;
          if (g == 0) {
            dst[0] = mref[j][e];
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
    const int into = cc.tile % a.chunk_tiles;
    chunk_left = min(a.chunk_tiles - into, cc.ntiles - cc.tile);
    if constexpr (kScl == kSclUnit) {
      const int si = cc.kvh * a.scale_head_stride;
      sc = __ldg(a.k_scales + si) * a.logit_scale;
      unit_vs = __ldg(a.v_scales + si);
    }
    if constexpr (kScl == kSclToken) {
      vref = 0.f;
      vinv = 0.f;
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      mref[j][0] = mref[j][1] = -INFINITY;
      rthr[j][0] = rthr[j][1] = -INFINITY;
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
      for (int i = 0; i < 16; ++i) qf[j][i >> 1][i & 1] = wd[i];  // bf16 pairs
    }
    if constexpr (!kBf16 && kScl == kSclToken) {
      // Q in f16 for the widened-K products, times a power of two s over the
      // unit's heads taking max |q s| into (2^14, 2^15]: every finite bf16
      // query fits and each value at least 2^-29 of the largest is an exact
      // f16 normal; the raw scores are multiplied by 1 / s
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int i = 0; i < 16; ++i)
          amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(qf[j][i >> 1][i & 1])), fabsf(bf16_hi(qf[j][i >> 1][i & 1]))));
#pragma unroll
      for (int o2 = 16; o2 >= 1; o2 >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o2));
      const float s = pow2_scale(32768.f, amax);
      qinv[0][0] = 1.f / s;  // exact: s is a power of two
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t w = qf[j][i >> 1][i & 1];
          qf[j][i >> 1][i & 1] = pack_f16x2(bf16_lo(w) * s, bf16_hi(w) * s);
        }
    } else if constexpr (!kBf16) {
      // Q as two exact e4m3 parts for the e4m3 products on the raw K bytes:
      // x = q s with s a power of two per head, s = 2^floor(log2(448 /
      // max |q|)) over the head's 128 values (the four lanes of group g hold
      // them); part 1 = e4m3(x), part 2 = e4m3(x - part 1): a bf16 value
      // has 8 significant bits, each part 4, so every scaled value above 1/4
      // (at least 1/896 of the head's largest) is split exactly, and smaller
      // ones within 2^-10.  Register pair (2 kk + p)
      // holds part p of head_dim values 32t + 8kk .. 32t + 8kk + 7, the K
      // elements that the e4m3 product's k 4t.. and 16 + 4t.. pick in step kk.
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(qf[j][i >> 1][i & 1])), fabsf(bf16_hi(qf[j][i >> 1][i & 1]))));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        const float s = pow2_scale(448.f, amax);
        const float hinv = 1.f / s;  // head 8j + g; exact: s is a power of two
        // the score columns of this thread are heads 8j + 2t and 8j + 2t + 1
        qinv[j][0] = __shfl_sync(0xFFFFFFFFu, hinv, 8 * t);
        qinv[j][1] = __shfl_sync(0xFFFFFFFFu, hinv, 8 * t + 4);
        uint32_t wq[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) wq[i] = qf[j][i >> 1][i & 1];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t p1[2], p2[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // bf16 pairs wq[4kk + 2h], wq[4kk + 2h + 1]: four values
            uint32_t c1w = 0u, c2w = 0u;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const uint32_t w = wq[4 * kk + 2 * h + e];
              const float x0 = bf16_lo(w) * s, x1 = bf16_hi(w) * s;
              const uint16_t c1 = f32x2_to_e4m3x2(x0, x1);
              const uint32_t hf = e4m3x2_to_f16x2(c1);
              const uint16_t c2 = f32x2_to_e4m3x2(x0 - f16_lo(hf), x1 - f16_hi(hf));  // exact difference
              c1w |= (uint32_t)c1 << (16 * e);
              c2w |= (uint32_t)c2 << (16 * e);
            }
            p1[h] = c1w;
            p2[h] = c2w;
          }
          qf[j][2 * kk][0] = p1[0];
          qf[j][2 * kk][1] = p1[1];
          qf[j][2 * kk + 1][0] = p2[0];
          qf[j][2 * kk + 1][1] = p2[1];
        }
      }
    }
  };

  int stage = 0;
  uint32_t phase = 0;
  int64_t f_stop_at = f_end;  // first tile not consumed (differs from f_end on a timeout)
  bool timed_out = false;
  bool need_start = true;
  for (int64_t f = f_begin; f < f_end; ++f) {
    if (need_start) {
      start_unit();
      seg_begin = f;
      need_start = false;
    }
    if (!mbar_wait(bar0 + 8 * stage, phase)) {
      timed_out = true;
      f_stop_at = f;
      break;
    }
    const uint8_t* kb = wptr + stage * Geo::kStageBytes;
    const uint8_t* vb = kb + Geo::kKBytes;
    const int tok0 = cc.tile * kTile;
    const bool partial = tok0 + kTile > L;  // warp-uniform: only the last tile of a request

    // ---------------- S^T = K . Q^T  (rows: tokens, cols: heads), raw units
    float s[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
    if constexpr (kBf16) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint8_t* hb = kb + h2 * 2048;
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
    } else if constexpr (kScl == kSclToken) {
      // per-token scales: K widened to f16 (this variant is at its register
      // limit, where the e4m3 products' Q parts cost more than they save)
      const uint4 x0 = lds128(kb + swz(g, 2 * t)), x1 = lds128(kb + swz(g, 2 * t + 1));
      const uint4 y0 = lds128(kb + swz(g + 8, 2 * t)), y1 = lds128(kb + swz(g + 8, 2 * t + 1));
      const uint32_t xr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t yr[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2x2(xr[ks], a0, a2);
        e4m3x4_to_f16x2x2(yr[ks], a1, a3);
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_f16(s[j], a0, a1, a2, a3, qf[j][ks][0], qf[j][ks][1]);
      }
    } else {
      const uint4 x0 = lds128(kb + swz(g, 2 * t)), x1 = lds128(kb + swz(g, 2 * t + 1));
      const uint4 y0 = lds128(kb + swz(g + 8, 2 * t)), y1 = lds128(kb + swz(g + 8, 2 * t + 1));
      const uint32_t xr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t yr[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
      // the K bytes feed the e4m3 products as they are: step kk takes head_dim
      // 32t + 8kk .. 32t + 8kk + 7 of rows g and g + 8, against Q's two parts
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          mma_e4m3(s[j], xr[2 * kk], yr[2 * kk], xr[2 * kk + 1], yr[2 * kk + 1], qf[j][2 * kk][0], qf[j][2 * kk][1]);
          mma_e4m3(s[j], xr[2 * kk], yr[2 * kk], xr[2 * kk + 1], yr[2 * kk + 1], qf[j][2 * kk + 1][0],
                   qf[j][2 * kk + 1][1]);
        }
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {  // undo the Q scale (a power of two: exact)
        s[j][0] *= qinv[j][0];
        s[j][1] *= qinv[j][1];
        s[j][2] *= qinv[j][0];
        s[j][3] *= qinv[j][1];
      }
    }

    // ---------------- per-token scales: this thread's tokens are g and g + 8
    float ks0 = 1.f, ks8 = 1.f, vs0 = 0.f, vs8 = 0.f;
    if constexpr (kScl == kSclToken) {
      const float* sp = sptr + stage * (kScaleStageBytes / 4);
      ks0 = sp[g] * qinv[0][0];  // the token's K scale and the Q scale's inverse
      ks8 = sp[g + 8] * qinv[0][0];
      vs0 = sp[16 + g];
      vs8 = sp[24 + g];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        s[j][0] *= ks0;
        s[j][1] *= ks0;
        s[j][2] *= ks8;
        s[j][3] *= ks8;
      }
    }

    // ---------------- mask (last tile only), lazy online softmax (exp2 domain)
    if (partial) {
      const bool va = tok0 + g < L, vb8 = tok0 + g + 8 < L;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        if (!va) s[j][0] = s[j][1] = -INFINITY;
        if (!vb8) s[j][2] = s[j][3] = -INFINITY;
      }
      if constexpr (kScl == kSclToken) {  // scales past the context are never used
        if (!va) vs0 = 0.f;
        if (!vb8) vs8 = 0.f;
      }
    }
    bool grow = false;
#pragma unroll
    for (int j = 0; j < NT; ++j)
      grow |= (fmaxf(s[j][0], s[j][2]) > rthr[j][0]) | (fmaxf(s[j][1], s[j][3]) > rthr[j][1]);
    if (__any_sync(0xFFFFFFFFu, grow)) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float mx0 = fmaxf(s[j][0], s[j][2]), mx1 = fmaxf(s[j][1], s[j][3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
        }
        const float mn0 = fmaxf(mref[j][0], mx0 * sc), mn1 = fmaxf(mref[j][1], mx1 * sc);
        const float al0 = fast_exp2(mref[j][0] - mn0), al1 = fast_exp2(mref[j][1] - mn1);
        l[j][0] *= al0;
        l[j][1] *= al1;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          o[j][i][0] *= al0;
          o[j][i][1] *= al1;
          o[j][i][2] *= al0;
          o[j][i][3] *= al1;
        }
        mref[j][0] = mn0;
        mref[j][1] = mn1;
        rthr[j][0] = (mn0 + kRescaleLog2) / sc;
        rthr[j][1] = (mn1 + kRescaleLog2) / sc;
      }
    }
    // per-token V scales enter as weights on p relative to vref, the largest V
    // scale of the unit so far, so that p * weight <= p stays in f16 range;
    // when vref grows the accumulator is rescaled like the running maximum
    float w0 = 1.f, w8 = 1.f;
    if constexpr (kScl == kSclToken) {
      // the largest V scale of the tile: with one or two heads per KV head the
      // tile's work is too short to hide a shuffle chain, so every thread
      // reads the tile's 16 V scales from the stage; with more heads the
      // chain is hidden and costs fewer instructions
      float vm;
      if (a.G <= 2) {
        const float4* vp = reinterpret_cast<const float4*>(sptr + stage * (kScaleStageBytes / 4) + 16);
        float4 q4[4] = {vp[0], vp[1], vp[2], vp[3]};
        if (partial) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (tok0 + 4 * i >= L) q4[i].x = 0.f;
            if (tok0 + 4 * i + 1 >= L) q4[i].y = 0.f;
            if (tok0 + 4 * i + 2 >= L) q4[i].z = 0.f;
            if (tok0 + 4 * i + 3 >= L) q4[i].w = 0.f;
          }
        }
        float m4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) m4[i] = fmaxf(fmaxf(q4[i].x, q4[i].y), fmaxf(q4[i].z, q4[i].w));
        vm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      } else {
        vm = fmaxf(vs0, vs8);
        vm = fmaxf(vm, __shfl_xor_sync(0xFFFFFFFFu, vm, 4));
        vm = fmaxf(vm, __shfl_xor_sync(0xFFFFFFFFu, vm, 8));
        vm = fmaxf(vm, __shfl_xor_sync(0xFFFFFFFFu, vm, 16));
      }
      if (vm > vref) {  // warp-uniform
        const float r = vref / vm;
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[j][i][0] *= r;
            o[j][i][1] *= r;
            o[j][i][2] *= r;
            o[j][i][3] *= r;
          }
        vref = vm;
        vinv = 1.f / vm;
      }
      w0 = vs0 * vinv;
      w8 = vs8 * vinv;
    }
    uint32_t pb[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      float p0 = fast_exp2(fmaf(s[j][0], sc, -mref[j][0]));
      float p1 = fast_exp2(fmaf(s[j][1], sc, -mref[j][1]));
      float p2 = fast_exp2(fmaf(s[j][2], sc, -mref[j][0]));
      float p3 = fast_exp2(fmaf(s[j][3], sc, -mref[j][1]));
      l[j][0] += p0 + p2;
      l[j][1] += p1 + p3;
      if constexpr (kScl == kSclToken) {
        p0 *= w0;
        p1 *= w0;
        p2 *= w8;
        p3 *= w8;
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
    // Rows past the context hold arbitrary bytes (even NaN codes); they are
    // zeroed so that p = 0 cannot meet a NaN in the MMA.
    if constexpr (kBf16) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint8_t* hb = vb + h2 * 2048;
        uint4 r0 = lds128(hb + swz(2 * t, g)), r1 = lds128(hb + swz(2 * t + 1, g));
        uint4 r2 = lds128(hb + swz(2 * t + 8, g)), r3 = lds128(hb + swz(2 * t + 9, g));
        if (partial) {
          const uint4 z = make_uint4(0, 0, 0, 0);
          if (tok0 + 2 * t >= L) r0 = z;
          if (tok0 + 2 * t + 1 >= L) r1 = z;
          if (tok0 + 2 * t + 8 >= L) r2 = z;
          if (tok0 + 2 * t + 9 >= L) r3 = z;
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
        if (tok0 + 2 * t >= L) r0 = z;
        if (tok0 + 2 * t + 1 >= L) r1 = z;
        if (tok0 + 2 * t + 8 >= L) r2 = z;
        if (tok0 + 2 * t + 9 >= L) r3 = z;
      }
      const uint32_t R0[4] = {r0.x, r0.y, r0.z, r0.w}, R1[4] = {r1.x, r1.y, r1.z, r1.w};
      const uint32_t R2[4] = {r2.x, r2.y, r2.z, r2.w}, R3[4] = {r3.x, r3.y, r3.z, r3.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
        uint32_t A0, A1, A2, A3;
        e4m3x4_to_f16x2x2(prmt(R0[i >> 1], R1[i >> 1], sel), A0, A1);
        e4m3x4_to_f16x2x2(prmt(R2[i >> 1], R3[i >> 1], sel), A2, A3);
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
    if (--chunk_left == 0 || f + 1 == f_end) {
      flush(f + 1);
      need_start = true;
    }
    cursor_next(cc, a);
  }

  if (timed_out) {
    if (lane == 0) atomicOr(a.status, kErrWaitTimeout);
    // let every copy still in flight land (bounded waits) before the CTA's
    // shared memory is released
    int st = stage;
    uint32_t ph = phase;
    for (int64_t k = 0; k < f_issue - f_stop_at; ++k) {
      (void)mbar_wait(bar0 + 8 * st, ph);
      if (++st == kStages) {
        st = 0;
        ph ^= 1u;
      }
    }
  }
}

// -------------------------------------------------------------- merge kernel
// One CTA per (request, KV head).  Its segments -- one per (chunk, covering
// warp) -- are enumerated in batches of chunks (threads find each chunk's first
// covering warp and segment count; a block scan numbers the segments in shared
// memory).  The G heads' partial states of one segment are contiguous, so a
// warp reads all of them with coalesced loads; warps split the segments and
// fold them with an online maximum per head, and warp e then combines the
// warps' states of head e with the log-sum-exp rule
//   M = max_k m_k,  out = sum_k 2^{m_k-M} o_k / sum_k 2^{m_k-M} l_k.
// One head of a unit without explicit chunks: its segments are the
// consecutive warps first .. last that covered it (one warp per tile when
// there are fewer tiles than warps).  The calling warp folds them, four
// segments' loads in flight at a time, and writes the head's output.
__device__ __forceinline__ void merge_unit_head(const DecodeArgs& a, int64_t ts, int ntiles, int64_t u0, int e,
                                                int64_t head, int lane) {
  const int64_t W = a.tile_start[a.B], N = a.nwarps;
  const int64_t first = owner_of(ts, W, N);
  const int64_t nseg = W >= N ? owner_of(ts + ntiles - 1, W, N) - first + 1 : ntiles;
  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t k0 = 0; k0 < nseg; k0 += 4) {
    float mk[4], lk[4];
    float4 ok[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t k = k0 + q;
      mk[q] = -INFINITY;
      lk[q] = 0.f;
      ok[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k < nseg) {
        const int64_t slot = (W >= N ? first + k : owner_of(ts + k, W, N)) + u0;
        if (slot < a.capacity) {
          const float* p = a.partials + (slot * a.G + e) * kPartialStride;
          mk[q] = p[0];
          lk[q] = p[1];
          ok[q] = reinterpret_cast<const float4*>(p + 4)[lane];
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (mk[q] == -INFINITY) continue;
      const float Mn = fmaxf(M, mk[q]);
      const float al = fast_exp2(M - Mn), wt = fast_exp2(mk[q] - Mn);
      den = den * al + wt * lk[q];
      acc.x = acc.x * al + wt * ok[q].x;
      acc.y = acc.y * al + wt * ok[q].y;
      acc.z = acc.z * al + wt * ok[q].z;
      acc.w = acc.w * al + wt * ok[q].w;
      M = Mn;
    }
  }
  const float inv = den > 0.f ? a.out_scale / den : 0.f;
  reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + head * kD)[lane] =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (a.lse && lane == 0) a.lse[head] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
}

constexpr int kMergeWarps = 8;
constexpr int kMergeThreads = kMergeWarps * 32;
constexpr int kMergeBatch = kMergeThreads;  // chunks enumerated per batch
constexpr int kMergeLoads = 4;              // segments per warp whose loads are in flight together

// kMergeHeads query heads of one (request, KV head) per CTA; calls with
// explicit chunks use 1 (many small CTAs), calls without them use
// merge_unsplit_kernel below.
template <int kMergeHeads>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const DecodeArgs a) {
  __shared__ float4 red_o[kMergeWarps][kMergeHeads][32];
  __shared__ float red_m[kMergeWarps][kMergeHeads], red_l[kMergeWarps][kMergeHeads];
  __shared__ int32_t seg_base[kMergeBatch + 1];
  __shared__ int32_t first_w[kMergeBatch];
  __shared__ int16_t seg_chunk[kMergeBatch + kMaxWarps];  // batch-local chunk of each segment
  __shared__ int32_t scan_tmp[kMergeWarps];
  grid_dependency_wait();  // every partial state of the tile kernel is visible
  const int groups = (a.G + kMergeHeads - 1) / kMergeHeads;
  const int bk = blockIdx.x / groups;
  const int g_lo = (blockIdx.x % groups) * kMergeHeads;  // first head of this CTA
  const int g_hi = min(a.G, g_lo + kMergeHeads);
  const int b = bk / a.Hkv, kvh = bk % a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t head0 = (int64_t)b * a.Hq + (int64_t)kvh * a.G;
  const int ntiles = ntiles_of(a, b);
  if (ntiles == 0) {
    for (int e = g_lo + warp; e < g_hi; e += kMergeWarps) {
      reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + (head0 + e) * kD)[lane] = make_uint2(0, 0);
      if (a.lse && lane == 0) a.lse[head0 + e] = -INFINITY;
    }
    return;
  }
  const int64_t W = a.tile_start[a.B], N = a.nwarps;
  const int nchunks = (int)((a.unit_start[b + 1] - a.unit_start[b]) / a.Hkv);
  const int64_t ts = a.tile_start[b] + (int64_t)kvh * ntiles;
  const int64_t u0 = a.unit_start[b] + (int64_t)kvh * nchunks;
  if (nchunks == 1 && owner_of(ts, W, N) == owner_of(ts + ntiles - 1, W, N)) return;  // direct
  if (nchunks == 1) {
    // one warp per head (with one head per CTA, warp 0)
    const int e = g_lo + (kMergeHeads == 1 ? 0 : warp);
    if ((kMergeHeads == 1 && warp != 0) || e >= g_hi) return;
    merge_unit_head(a, ts, ntiles, u0, e, head0 + e, lane);
    return;
  }

  {
    const int e0 = g_lo;
    const int ne = g_hi - g_lo;
    float M[kMergeHeads], den[kMergeHeads];
    float4 acc[kMergeHeads];
#pragma unroll
    for (int e = 0; e < kMergeHeads; ++e) {
      M[e] = -INFINITY;
      den[e] = 0.f;
      acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int c0 = 0; c0 < nchunks; c0 += kMergeBatch) {
      const int nb = min(kMergeBatch, nchunks - c0);
      // ---- enumerate this batch's segments
      int32_t nseg = 0;
      if (threadIdx.x < nb) {
        const int c = c0 + threadIdx.x;
        const int64_t s_c = ts + (int64_t)c * a.chunk_tiles;
        const int64_t e_c = min(s_c + (int64_t)a.chunk_tiles, ts + ntiles);
        const int64_t first = owner_of(s_c, W, N), last = owner_of(e_c - 1, W, N);
        // W >= N: every warp owns tiles, owners are consecutive; W < N: one tile per warp
        nseg = (int32_t)(W >= N ? last - first + 1 : e_c - s_c);
        first_w[threadIdx.x] = (int32_t)first;
      }
      int32_t x = nseg;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) scan_tmp[warp] = x;
      __syncthreads();
      int32_t pre = 0;
      for (int k = 0; k < warp; ++k) pre += scan_tmp[k];
      if (threadIdx.x < nb) {
        seg_base[threadIdx.x] = pre + x - nseg;
        for (int32_t k = 0; k < nseg; ++k)
          if (pre + x - nseg + k < kMergeBatch + kMaxWarps)
            seg_chunk[pre + x - nseg + k] = (int16_t)threadIdx.x;
      }
      if (threadIdx.x == kMergeThreads - 1) seg_base[nb] = pre + x;
      __syncthreads();
      const int32_t total = min(seg_base[nb], (int32_t)(kMergeBatch + kMaxWarps));
      // ---- fold: warps stride over segments, kMergeLoads of them per round
      // with every load issued before the first fold; lane l owns head_dim
      // 4l..4l+3
      for (int32_t sg0 = warp; sg0 < total; sg0 += kMergeWarps * kMergeLoads) {
        float mk[kMergeLoads][kMergeHeads], lk[kMergeLoads][kMergeHeads];
        float4 ok[kMergeLoads][kMergeHeads];
#pragma unroll
        for (int r = 0; r < kMergeLoads; ++r) {
          const int32_t sg = sg0 + r * kMergeWarps;
#pragma unroll
          for (int e = 0; e < kMergeHeads; ++e) {
            mk[r][e] = -INFINITY;
            lk[r][e] = 0.f;
            ok[r][e] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          if (sg >= total) continue;
          const int lo = seg_chunk[sg];
          const int32_t k = sg - seg_base[lo];
          const int c = c0 + lo;
          const int64_t w = W >= N ? (int64_t)first_w[lo] + k
                                   : owner_of(ts + (int64_t)c * a.chunk_tiles + k, W, N);
          const int64_t slot = w + u0 + c;
          if (slot >= a.capacity) continue;
          const float* p = a.partials + (slot * a.G + e0) * kPartialStride;
#pragma unroll
          for (int e = 0; e < kMergeHeads; ++e) {
            if (e < ne) {
              mk[r][e] = p[e * kPartialStride];
              lk[r][e] = p[e * kPartialStride + 1];
              ok[r][e] = reinterpret_cast<const float4*>(p + e * kPartialStride + 4)[lane];
            }
          }
        }
#pragma unroll
        for (int r = 0; r < kMergeLoads; ++r)
#pragma unroll
          for (int e = 0; e < kMergeHeads; ++e) {
            if (e >= ne || mk[r][e] == -INFINITY) continue;
            const float Mn = fmaxf(M[e], mk[r][e]);
            const float al = fast_exp2(M[e] - Mn), wt = fast_exp2(mk[r][e] - Mn);
            den[e] = den[e] * al + wt * lk[r][e];
            acc[e].x = acc[e].x * al + wt * ok[r][e].x;
            acc[e].y = acc[e].y * al + wt * ok[r][e].y;
            acc[e].z = acc[e].z * al + wt * ok[r][e].z;
            acc[e].w = acc[e].w * al + wt * ok[r][e].w;
            M[e] = Mn;
          }
        // The states just folded are dead: drop their lines from L2 without
        // writing them back (left dirty, their write-back would compete with
        // the next call's K/V stream for HBM; measured: 1,817-1,828 -> 1,783 us
        // per call back to back on 8 requests of 256K-1M tokens).  With one
        // head per CTA no other CTA reads these five lines.
        __syncwarp();  // every lane's loads of these states have completed
        if (kMergeHeads == 1 && lane < kPartialStride / 32) {
#pragma unroll
          for (int r = 0; r < kMergeLoads; ++r) {
            const int32_t sg = sg0 + r * kMergeWarps;
            if (sg >= total) continue;
            const int lo = seg_chunk[sg];
            const int32_t k = sg - seg_base[lo];
            const int c = c0 + lo;
            const int64_t w = W >= N ? (int64_t)first_w[lo] + k
                                     : owner_of(ts + (int64_t)c * a.chunk_tiles + k, W, N);
            const int64_t slot = w + u0 + c;
            if (slot >= a.capacity) continue;
            l2_discard_line(a.partials + (slot * a.G + e0) * kPartialStride + 32 * lane);
          }
        }
      }
      __syncthreads();  // seg_base / first_w / seg_chunk are rewritten by the next batch
    }
    // ---- combine the warps' states; warp e finishes head e0 + e
#pragma unroll
    for (int e = 0; e < kMergeHeads; ++e) {
      red_o[warp][e][lane] = acc[e];
      if (lane == 0) {
        red_m[warp][e] = M[e];
        red_l[warp][e] = den[e];
      }
    }
    __syncthreads();
    if (warp < ne) {
      const int e = warp;
      float Mt = -INFINITY;
#pragma unroll
      for (int k = 0; k < kMergeWarps; ++k) Mt = fmaxf(Mt, red_m[k][e]);
      float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
      float dt = 0.f;
#pragma unroll
      for (int k = 0; k < kMergeWarps; ++k) {
        if (red_m[k][e] == -INFINITY) continue;
        const float wt = fast_exp2(red_m[k][e] - Mt);
        const float4 v = red_o[k][e][lane];
        tot.x += wt * v.x;
        tot.y += wt * v.y;
        tot.z += wt * v.z;
        tot.w += wt * v.w;
        dt += wt * red_l[k][e];
      }
      const int64_t head = head0 + e0 + e;
      const float inv = a.out_scale / dt;
      reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + head * kD)[lane] =
          make_uint2(pack_bf16x2(tot.x * inv, tot.y * inv), pack_bf16x2(tot.z * inv, tot.w * inv));
      if (a.lse && lane == 0) a.lse[head] = (Mt + __log2f(dt)) * kLn2;
    }
  }
}

// Merge for calls without explicit chunks (one unit per request and KV head):
// one warp per (request, query head), eight per CTA, so that every unit's
// heads are folded in a single wave of small CTAs.
__global__ void __launch_bounds__(kMergeThreads) merge_unsplit_kernel(const DecodeArgs a) {
  grid_dependency_wait();  // every partial state of the tile kernel is visible
  const int64_t hw = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);  // b * Hq + query head
  const int lane = threadIdx.x & 31;
  if (hw >= (int64_t)a.B * a.Hq) return;
  const int b = (int)(hw / a.Hq), hq = (int)(hw % a.Hq);
  const int kvh = hq / a.G, e = hq % a.G;
  const int ntiles = ntiles_of(a, b);
  if (ntiles == 0) {
    reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + hw * kD)[lane] = make_uint2(0, 0);
    if (a.lse && lane == 0) a.lse[hw] = -INFINITY;
    return;
  }
  const int64_t W = a.tile_start[a.B], N = a.nwarps;
  const int64_t ts = a.tile_start[b] + (int64_t)kvh * ntiles;
  if (owner_of(ts, W, N) == owner_of(ts + ntiles - 1, W, N)) return;  // one warp wrote it directly
  merge_unit_head(a, ts, ntiles, a.unit_start[b] + kvh, e, hw, lane);
}

// ------------------------------------------------------------------- host
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t tile_off, unit_off, part_off;
};

// Bytes per partial slot: the fp32 states of G heads.
size_t slot_bytes(int G) { return (size_t)G * kPartialStride * sizeof(float); }

WsLayout ws_layout(int B) {
  WsLayout L;
  L.tile_off = 256;
  L.unit_off = align_up(L.tile_off + sizeof(int64_t) * (size_t)(B + 1), 256);
  L.part_off = align_up(L.unit_off + sizeof(int64_t) * (size_t)(B + 1), 256);
  return L;
}

template <bool kBf16, int NT, int kScl>
int launch_decode(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeArgs& a,
                  cudaStream_t stream) {
  using Geo = Geometry<kBf16, kScl>;
  auto kern = paged_decode_kernel<kBf16, NT, kScl>;
  static std::atomic<uint64_t> smem_set{0};
  const int rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), Geo::kSmemBytes, smem_set,
                                      "paged_decode set smem attribute");
  if (rc != PFKV_OK) return rc;
  // persistent grid: every SM filled with resident CTAs (cached per device)
  static int grid_of_device[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return check_cuda("paged_decode cudaGetDevice");
  int grid = (dev >= 0 && dev < 64) ? grid_of_device[dev] : 0;
  if (grid == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, Geo::kSmemBytes) !=
        cudaSuccess)
      return check_cuda("paged_decode occupancy");
    if (per_sm < 1) per_sm = 1;
    grid = device_sm_count() * per_sm;
    if (grid < 1) grid = 1;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (dev >= 0 && dev < 64) grid_of_device[dev] = grid;
  }
  DecodeArgs args = a;
  args.nwarps = (int64_t)grid * kWarps;
  plan_kernel<<<1, 1024, 0, stream>>>(args);
  // the tile kernel and the merge kernel are launched as programmatic
  // dependents, so their launch overlaps the tail of the kernel before them;
  // each waits (griddepcontrol.wait) before reading what that kernel wrote
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = Geo::kSmemBytes;
  if (cudaLaunchKernelEx(&cfg, kern, tmK, tmV, args) != cudaSuccess) return check_cuda("paged_decode launch");
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cudaError_t e;
  if (a.chunk_tiles < (1 << 30)) {
    cfg.gridDim = dim3(a.B * a.Hq);
    e = cudaLaunchKernelEx(&cfg, merge_kernel<1>, args);
  } else {
    cfg.gridDim = dim3((unsigned)(((int64_t)a.B * a.Hq + kMergeWarps - 1) / kMergeWarps));
    e = cudaLaunchKernelEx(&cfg, merge_unsplit_kernel, args);
  }
  if (e != cudaSuccess) return check_cuda("paged_decode merge launch");
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
  return L.part_off + (size_t)slots * pfkv::slot_bytes(G) + 1024;
}

}  // extern "C"

namespace pfkv {
namespace {

// The decode entry for every scale mode: kSclHost takes k_scale / v_scale;
// kSclUnit and kSclToken read the device arrays k_scales / v_scales (unit
// mode: one scale per KV head when head_stride is 1, one for all when 0).
int decode_entry(void* out, const void* q, const void* k_cache, const void* v_cache,
                 pfkv_cache_dtype cache_dtype, const int32_t* block_tables, int max_pages_per_seq,
                 const int32_t* context_lens, int batch, int num_q_heads, int num_kv_heads,
                 int head_dim, int page_size, int64_t num_pages, float k_scale, float v_scale,
                 float softmax_scale, int kv_split_tokens, void* workspace, size_t workspace_bytes,
                 float* lse_out, pfkv_stream_t stream, int scl, const float* k_scales,
                 const float* v_scales, int head_stride) {
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
  if (scl != kSclHost) {
    if (cache_dtype != PFKV_CACHE_FP8_E4M3)
      return fail(PFKV_ERR_UNSUPPORTED, "paged_decode_scaled: device scales need the e4m3 cache");
    if (!k_scales || !v_scales) return fail(PFKV_ERR_INVALID_ARG, "paged_decode_scaled: null scale array");
    if (!aligned(k_scales, 16) || !aligned(v_scales, 16))
      return fail(PFKV_ERR_INVALID_ARG, "paged_decode_scaled: scale arrays must be 16-byte aligned");
  }
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
  if (workspace_bytes <
      L.part_off + slot_bytes(G) * ((size_t)kMaxWarps + (size_t)num_kv_heads * batch) + 1024)
    return fail(PFKV_ERR_WORKSPACE, "paged_decode: workspace of %zu bytes is too small",
                workspace_bytes);
  const int64_t cap = (int64_t)((workspace_bytes - L.part_off - 1024) / slot_bytes(G));

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
  a.capacity = cap;
  a.nwarps = 0;
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
  a.k_scales = k_scales;
  a.v_scales = v_scales;
  a.scale_head_stride = head_stride;
  a.logit_scale = softmax_scale * kLog2e;
  if (scl != kSclHost) {  // the device scales carry K and V; the merge multiplies by 1
    a.score_scale = a.logit_scale;
    a.out_scale = 1.f;
  }

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
    return G <= 8 ? launch_decode<true, 1, kSclHost>(tmK, tmV, a, s)
                  : launch_decode<true, 2, kSclHost>(tmK, tmV, a, s);
  if (scl == kSclUnit)
    return G <= 8 ? launch_decode<false, 1, kSclUnit>(tmK, tmV, a, s)
                  : launch_decode<false, 2, kSclUnit>(tmK, tmV, a, s);
  if (scl == kSclToken)
    return G <= 8 ? launch_decode<false, 1, kSclToken>(tmK, tmV, a, s)
                  : launch_decode<false, 2, kSclToken>(tmK, tmV, a, s);
  return G <= 8 ? launch_decode<false, 1, kSclHost>(tmK, tmV, a, s)
                : launch_decode<false, 2, kSclHost>(tmK, tmV, a, s);
}

}  // namespace
}  // namespace pfkv

extern "C" {

int pfkv_paged_decode_attn(void* out, const void* q, const void* k_cache, const void* v_cache,
                           pfkv_cache_dtype cache_dtype, const int32_t* block_tables,
                           int max_pages_per_seq, const int32_t* context_lens, int batch,
                           int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                           int64_t num_pages, float k_scale, float v_scale, float softmax_scale,
                           int kv_split_tokens, void* workspace, size_t workspace_bytes,
                           float* lse_out, pfkv_stream_t stream) {
  return pfkv::decode_entry(out, q, k_cache, v_cache, cache_dtype, block_tables, max_pages_per_seq,
                            context_lens, batch, num_q_heads, num_kv_heads, head_dim, page_size,
                            num_pages, k_scale, v_scale, softmax_scale, kv_split_tokens, workspace,
                            workspace_bytes, lse_out, stream, pfkv::kSclHost, nullptr, nullptr, 0);
}

int pfkv_paged_decode_attn_scaled(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  pfkv_scale_granularity granularity, const float* k_scales,
                                  const float* v_scales, const int32_t* block_tables,
                                  int max_pages_per_seq, const int32_t* context_lens, int batch,
                                  int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                                  int64_t num_pages, float softmax_scale, int kv_split_tokens,
                                  void* workspace, size_t workspace_bytes, float* lse_out,
                                  pfkv_stream_t stream) {
  using namespace pfkv;
  int scl, stride = 0;
  switch (granularity) {
    case PFKV_SCALE_TENSOR: scl = kSclUnit; break;
    case PFKV_SCALE_HEAD: scl = kSclUnit; stride = 1; break;
    case PFKV_SCALE_TOKEN: scl = kSclToken; break;
    default:
      clear_error();
      return fail(PFKV_ERR_INVALID_ARG, "paged_decode_scaled: unknown granularity %d", (int)granularity);
  }
  return decode_entry(out, q, k_cache, v_cache, PFKV_CACHE_FP8_E4M3, block_tables, max_pages_per_seq,
                      context_lens, batch, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                      1.f, 1.f, softmax_scale, kv_split_tokens, workspace, workspace_bytes, lse_out,
                      stream, scl, k_scales, v_scales, stride);
}

}  // extern "C"

// --------------------------------------------------- no-allocation variant
// Some callers cannot allocate device memory at the point where they run
// decode: a serving engine that reserves the whole device up front and owns
// every byte through its own pool, or a per-token path that must not take the
// synchronisation and latency of cudaMalloc.  For them the scratch that
// paged_decode_attn needs lives in one file-scope device array of fixed size
// that is part of the loaded module; each GPU that loads this library keeps
// it until the process exits.
#include <mutex>

namespace pfkv {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;  // 64 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  The host-side
// name of the array is only a stand-in: the address must come from the
// runtime, once per device, with that device current.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return check_cuda("paged_decode_attn_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return fail(PFKV_ERR_UNSUPPORTED, "paged_decode_attn_noalloc: device %d beyond %d", dev,
                kNoAllocMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(PFKV_ERR_CUDA, "paged_decode_attn_noalloc: cudaGetSymbolAddress failed: %s",
                  cudaGetErrorString(e));
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return PFKV_OK;
}

}  // namespace
}  // namespace pfkv

extern "C" int pfkv_paged_decode_attn_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache, pfkv_cache_dtype cache_dtype,
    const int32_t* block_tables, int max_pages_per_seq, const int32_t* context_lens, int batch,
    int num_q_heads, int num_kv_heads, int head_dim, int page_size, int64_t num_pages, float k_scale,
    float v_scale, float softmax_scale, int kv_split_tokens, int64_t max_total_chunks, float* lse_out,
    int32_t* status_out, pfkv_stream_t stream) {
  using namespace pfkv;
  clear_error();
  const size_t need = pfkv_paged_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                       kv_split_tokens, max_total_chunks);
  if (need == 0)
    return fail(PFKV_ERR_INVALID_ARG, "paged_decode_attn_noalloc: bad batch or head counts");
  if (need > kNoAllocScratchBytes)
    return fail(PFKV_ERR_WORKSPACE,
                "paged_decode_attn_noalloc: this call needs %zu bytes of scratch; the built-in "
                "scratch holds %zu bytes (64 MiB) -- use pfkv_paged_decode_attn with a workspace",
                need, kNoAllocScratchBytes);
  void* ws = nullptr;
  int rc = noalloc_scratch(&ws);
  if (rc != PFKV_OK) return rc;
  // The decode path itself zeroes the status word at the start of the
  // scratch and writes every other scratch byte it later reads, so the
  // contents left by the previous call need no clearing here.
  rc = pfkv_paged_decode_attn(out, q, k_cache, v_cache, cache_dtype, block_tables, max_pages_per_seq,
                              context_lens, batch, num_q_heads, num_kv_heads, head_dim, page_size,
                              num_pages, k_scale, v_scale, softmax_scale, kv_split_tokens, ws,
                              kNoAllocScratchBytes, lse_out, stream);
  if (rc != PFKV_OK || status_out == nullptr) return rc;
  if (batch == 0) {  // nothing was enqueued: the status of an empty call is 0
    if (cudaMemsetAsync(status_out, 0, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return check_cuda("paged_decode_attn_noalloc: status clear");
    return PFKV_OK;
  }
  if (cudaMemcpyAsync(status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return check_cuda("paged_decode_attn_noalloc: status copy");
  return PFKV_OK;
}
