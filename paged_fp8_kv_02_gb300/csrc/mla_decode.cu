// mla_decode.cu -- MLA absorbed-latent decode over one shared e4m3 latent row
// per token, optionally restricted to a top-k token list.
//
// kLLM article (快手万擎大模型推理成本和性能优化实践), §5.1.1: DSA selects the
// top-k historical tokens that take part in attention and MLA stores a
// compressed per-token latent cKV; §5.1.2: that latent is shared by all heads
// (it cannot be split by head the way GQA KV heads can).  Absorbed reading: the
// whole Dqk = 576-wide row is the key, its first 512 entries are the value.
//
// Kernel: one CTA per (request, 32 query heads).  A producer warp gathers the
// 64 latent rows of each token tile straight from their pages with bulk copies
// (cp.async.bulk, one 576-byte row each) into a ring of shared-memory stages;
// the consumer warps run both contractions on warp-level tensor-core MMA
// (m16n8k16, f32 accumulate) with the e4m3 -> f16 conversion fused into the
// fragment build:
//   S[32 heads x 64 tokens] = Q . C^T  (K = 576; the head_dim sum is permuted
//                                       consistently in Q and in C's fragments)
//   O[32 heads x 512]      += P . C[:, 0:512]
// with an exp2 online softmax whose reference maximum is only raised when a
// score exceeds it by more than 2^8 (an exact re-parametrisation).  Sixteen
// consumer warps: for the scores each owns a 16-head x 8-token tile, for the
// output 32 columns of all 32 heads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "pfkv_internal.h"
#include "pfkv_ptx.cuh"

namespace pfkv {
namespace {

constexpr int kDqk = 576, kDv = 512;
constexpr int kHeads = 32;                    // query heads per CTA (2 MMA row tiles)
constexpr int kTok = 64;                      // tokens per tile
constexpr int kStages = 3;                    // latent-row ring depth
constexpr int kConsumers = 16;                // MMA warps
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kRowBytes = 592;                // staged row stride (576 + 16: bank spread)
constexpr int kStageBytes = kTok * kRowBytes;
constexpr int kQStride = kDqk * 2 + 16;       // bytes per staged Q row (f16, padded)
constexpr int kPStride = kTok * 2 + 16;       // bytes per P row (f16, padded)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;

constexpr int kSmemQ = kHeads * kQStride;                 // 37,376
constexpr int kSmemRows = kStages * kStageBytes;          // 113,664
constexpr int kSmemP = kHeads * kPStride;                 //  4,608
constexpr int kMaxRows = 2048;                            // rows resolved per pass
constexpr int kSmemSrc = kMaxRows * 8;                    // 16,384: row offsets (or -1)
constexpr size_t kSmemBytes = (size_t)kSmemQ + kSmemRows + kSmemP + kSmemSrc + 128;

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

// head_dim index of fragment k-index kk (0..15) in k-step s (0..35): within each
// 128-wide block thread t of a quad owns 32 contiguous bytes (16 in the last,
// 64-wide block), four per k-step: k = 2t, 2t+1, 2t+8, 2t+9 -> bytes 0..3.
__device__ __forceinline__ int perm_d(int s, int kk) {
  const int t = (kk & 7) >> 1;
  const int j = (kk & 1) | ((kk >> 3) << 1);
  if (s < 32) return 128 * (s >> 3) + 32 * t + 4 * (s & 7) + j;
  return 512 + 16 * t + 4 * (s - 32) + j;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void bulk_row(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) mla_decode_kernel(const MlaArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* qs = smem;                                  // [32][kQStride] f16, permuted head_dim
  uint8_t* rows = smem + kSmemQ;                       // [kStages][64][kRowBytes] e4m3
  uint8_t* ps = rows + kSmemRows;                      // [32][kPStride] f16
  int64_t* srcs = reinterpret_cast<int64_t*>(ps + kSmemP);  // [kMaxRows] cache row, -1 if none
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ int valid[kStages][kTok];
  __shared__ float red_max[2][8][16], red_l[2][8][16], alpha[kHeads];
  __shared__ int grow_flag;

  const int b = blockIdx.x, h0 = blockIdx.y * kHeads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  int L = a.context_lens[b];
  if (L < 0) L = 0;
  if (L > a.max_pages * a.P) L = a.max_pages * a.P;
  const int n = a.topk ? a.topk_n : L;
  const int ntiles = (n + kTok - 1) / kTok;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kConsumers);
    }
    fence_mbar_init();
  }
  // stage Q (bf16 -> f16) with the head_dim permutation used by the fragments
  for (int i = threadIdx.x; i < kHeads * kDqk; i += kThreads) {
    const int hr = i / kDqk, c = i % kDqk;  // c = 16 s + kk
    const int d = perm_d(c >> 4, c & 15);
    const int head = h0 + hr;
    float v = 0.f;
    if (head < a.H)
      v = __bfloat162float(a.q[((int64_t)b * a.H + head) * kDqk + d]);
    reinterpret_cast<__half*>(qs + hr * kQStride)[c] = __float2half_rn(v);
  }
  __syncthreads();

  bool timed_out = false;
  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    // Rows are resolved (top-k index -> block-table entry -> cache row) for
    // up to kMaxRows tokens at a time with independent loads from all lanes,
    // so the gather loop below only waits for free stages and issues copies.
    uint32_t ph_empty = 1;  // a fresh barrier's preceding phase counts as complete
    for (int it = 0; it < ntiles; ++it) {
      const int t0 = it * kTok;
      if (t0 % kMaxRows == 0) {
        __syncwarp();
        for (int r = lane; r < kMaxRows && t0 + r < n; r += 32) {
          const int tok = a.topk ? a.topk[(int64_t)b * a.topk_n + t0 + r] : t0 + r;
          int64_t row = -1;
          if (tok >= L && a.topk) atomicOr(a.status, kErrBadTopk);
          if (tok >= 0 && tok < L) {
            const int page = a.block_tables[(int64_t)b * a.max_pages + tok / a.P];
            if (page < 0 || (int64_t)page >= a.num_pages)
              atomicOr(a.status, kErrBadPage);
            else
              row = (int64_t)page * a.P + tok % a.P;
          }
          srcs[r] = row;
        }
        __syncwarp();
      }
      const int st = it % kStages;
      if (it > 0 && st == 0) ph_empty ^= 1u;
      if (!mbar_wait(smem_u32(&empty_bar[st]), ph_empty)) {
        timed_out = true;
        break;
      }
      uint8_t* sbase = rows + st * kStageBytes;
      int64_t srow[2];
      bool ok[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int r = lane + 32 * k;
        srow[k] = (t0 + r < n) ? srcs[(t0 + r) % kMaxRows] : -1;
        ok[k] = srow[k] >= 0;
        valid[st][r] = ok[k];
        if (!ok[k]) {  // rows that take no part are zero, so that p = 0 meets no NaN
          uint4* z = reinterpret_cast<uint4*>(sbase + r * kRowBytes);
          for (int w = 0; w < kDqk / 16; ++w) z[w] = make_uint4(0, 0, 0, 0);
        }
      }
      const uint32_t cnt = __popc(__ballot_sync(0xFFFFFFFFu, ok[0])) + __popc(__ballot_sync(0xFFFFFFFFu, ok[1]));
      fence_proxy_async_smem();  // zero rows (generic stores) before later bulk copies
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(smem_u32(&full_bar[st]), cnt * kDqk);
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (ok[k])
          bulk_row(smem_u32(sbase + (lane + 32 * k) * kRowBytes), a.ckv + srow[k] * kDqk, kDqk,
                   smem_u32(&full_bar[st]));
    }
    if (timed_out && lane == 0) atomicOr(a.status, kErrWaitTimeout);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int mt = warp & 1, nt = warp >> 1;  // scores: head tile, 8-token column tile
  const float sc = a.score_scale;
  float mref[2] = {-INFINITY, -INFINITY};  // rows g, g+8 of head tile mt
  float rthr[2] = {-INFINITY, -INFINITY};
  float lpart[2] = {0.f, 0.f};
  float o[2][4][4];  // [head tile][n-tile of this warp's 32 columns][frag]
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[i][j][0] = o[i][j][1] = o[i][j][2] = o[i][j][3] = 0.f;
  const uint32_t qs_u = smem_u32(qs), ps_u = smem_u32(ps);
  // ldmatrix row address of this lane for a 16x16 tile at (row0, col0 halves)
  const int lm_row = (lane & 7) + ((lane >> 3) & 1) * 8, lm_col = (lane >> 4) * 8;

  uint32_t ph_full = 0;
  for (int it = 0; it < ntiles; ++it) {
    const int st = it % kStages;
    if (it > 0 && st == 0) ph_full ^= 1u;
    // Every consumer warp runs the same sequence of named barriers whatever
    // happens: after a timed-out wait a warp stops waiting (and computes on
    // whatever the stage holds; the status word reports it) but keeps
    // iterating, so no warp is ever left at a barrier the others skipped.
    if (!timed_out && !mbar_wait(smem_u32(&full_bar[st]), ph_full)) timed_out = true;
    const uint8_t* sb = rows + st * kStageBytes;

    // ---- S = Q . C^T for head tile mt, tokens 8 nt .. 8 nt + 7; four
    // interleaved partial accumulators keep the MMA dependency chains short
    float sacc[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) sacc[k][0] = sacc[k][1] = sacc[k][2] = sacc[k][3] = 0.f;
    const uint8_t* r0 = sb + (8 * nt + g) * kRowBytes;
    const uint32_t qa = qs_u + (16 * mt + lm_row) * kQStride + lm_col * 2;
    uint32_t an[4];  // A fragment of the next k-step, loaded one step ahead
    ldmatrix_x4(qa, an[0], an[1], an[2], an[3]);
#pragma unroll
    for (int blk = 0; blk < 5; ++blk) {
      const int nsteps = blk < 4 ? 8 : 4;
      const int off = blk < 4 ? 128 * blk + 32 * t : 512 + 16 * t;
      uint32_t w0[8];
      {
        const uint4 x = *reinterpret_cast<const uint4*>(r0 + off);
        w0[0] = x.x; w0[1] = x.y; w0[2] = x.z; w0[3] = x.w;
      }
      if (blk < 4) {
        const uint4 x = *reinterpret_cast<const uint4*>(r0 + off + 16);
        w0[4] = x.x; w0[5] = x.y; w0[6] = x.z; w0[7] = x.w;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= nsteps) break;
        const int ks = (blk < 4 ? 8 * blk : 32) + j;
        const uint32_t a0 = an[0], a1 = an[1], a2 = an[2], a3 = an[3];
        if (ks + 1 < kDqk / 16) ldmatrix_x4(qa + 32 * (ks + 1), an[0], an[1], an[2], an[3]);
        uint32_t b0, b1;
        e4m3x4_to_f16x2x2(w0[j], b0, b1);
        mma_f16(sacc[ks & 3], a0, a1, a2, a3, b0, b1);
      }
    }
    float s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) s[e] = (sacc[0][e] + sacc[1][e]) + (sacc[2][e] + sacc[3][e]);

    // ---- mask, tile maximum across the eight column tiles, lazy rescale
    const int* vld = valid[st];
    {
      const int c0 = 8 * nt + 2 * t;
      if (!vld[c0]) s[0] = s[2] = -INFINITY;
      if (!vld[c0 + 1]) s[1] = s[3] = -INFINITY;
    }
    float mx0 = fmaxf(s[0], s[1]);  // row g
    float mx1 = fmaxf(s[2], s[3]);  // row g + 8
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
    }
    if (t == 0) {
      red_max[mt][nt][g] = mx0;
      red_max[mt][nt][g + 8] = mx1;
    }
    if (threadIdx.x == 0) grow_flag = 0;
    consumer_sync();
    float tm0 = red_max[mt][0][g], tm1 = red_max[mt][0][g + 8];
#pragma unroll
    for (int k = 1; k < 8; ++k) {
      tm0 = fmaxf(tm0, red_max[mt][k][g]);
      tm1 = fmaxf(tm1, red_max[mt][k][g + 8]);
    }
    float al0 = 1.f, al1 = 1.f;
    if (tm0 > rthr[0] || tm1 > rthr[1]) {  // identical in every warp of this head tile
      const float mn0 = fmaxf(mref[0], tm0 * sc), mn1 = fmaxf(mref[1], tm1 * sc);
      al0 = fast_exp2(mref[0] - mn0);
      al1 = fast_exp2(mref[1] - mn1);
      mref[0] = mn0;
      mref[1] = mn1;
      rthr[0] = (mn0 + kRescaleLog2) / sc;
      rthr[1] = (mn1 + kRescaleLog2) / sc;
      lpart[0] *= al0;
      lpart[1] *= al1;
      if (nt == 0 && t == 0) grow_flag = 1;
    }
    if (nt == 0 && t == 0) {
      alpha[16 * mt + g] = al0;
      alpha[16 * mt + g + 8] = al1;
    }
    // ---- P = 2^(s*scale - ref) -> f16 tile [head][token]
    {
      const float p0 = fast_exp2(fmaf(s[0], sc, -mref[0]));
      const float p1 = fast_exp2(fmaf(s[1], sc, -mref[0]));
      const float p2 = fast_exp2(fmaf(s[2], sc, -mref[1]));
      const float p3 = fast_exp2(fmaf(s[3], sc, -mref[1]));
      lpart[0] += p0 + p1;
      lpart[1] += p2 + p3;
      const int col = 8 * nt + 2 * t;
      *reinterpret_cast<uint32_t*>(ps + (16 * mt + g) * kPStride + col * 2) = pack_f16x2(p0, p1);
      *reinterpret_cast<uint32_t*>(ps + (16 * mt + g + 8) * kPStride + col * 2) = pack_f16x2(p2, p3);
    }
    consumer_sync();

    // ---- O[:, 32 w .. 32 w + 31] += P . C  (both head tiles)
    if (grow_flag) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float a_lo = alpha[16 * i + g], a_hi = alpha[16 * i + g + 8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          o[i][j][0] *= a_lo;
          o[i][j][1] *= a_lo;
          o[i][j][2] *= a_hi;
          o[i][j][3] *= a_hi;
        }
      }
    }
#pragma unroll
    for (int kstep = 0; kstep < kTok / 16; ++kstep) {
      uint32_t pa[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
        ldmatrix_x4(ps_u + (16 * i + lm_row) * kPStride + (16 * kstep + lm_col) * 2, pa[i][0], pa[i][1],
                    pa[i][2], pa[i][3]);
      // rows (tokens) 2t, 2t+1, 2t+8, 2t+9 of this k-step, 4 bytes at head_dim 32 w + 4 g:
      // n-tile j column g <-> head_dim 32 w + 4 g + j
      const uint8_t* base = sb + (16 * kstep) * kRowBytes + 32 * warp + 4 * g;
      const uint32_t v0 = *reinterpret_cast<const uint32_t*>(base + (2 * t) * kRowBytes);
      const uint32_t v1 = *reinterpret_cast<const uint32_t*>(base + (2 * t + 1) * kRowBytes);
      const uint32_t v2 = *reinterpret_cast<const uint32_t*>(base + (2 * t + 8) * kRowBytes);
      const uint32_t v3 = *reinterpret_cast<const uint32_t*>(base + (2 * t + 9) * kRowBytes);
      uint32_t bl[4], bh[4];  // b0b1 (tokens 2t, 2t+1) and b2b3 (tokens 2t+8, 2t+9) per n-tile
      e4m3x4_to_f16x2x2(prmt(v0, v1, 0x5140), bl[0], bl[1]);
      e4m3x4_to_f16x2x2(prmt(v0, v1, 0x7362), bl[2], bl[3]);
      e4m3x4_to_f16x2x2(prmt(v2, v3, 0x5140), bh[0], bh[1]);
      e4m3x4_to_f16x2x2(prmt(v2, v3, 0x7362), bh[2], bh[3]);
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_f16(o[i][j], pa[i][0], pa[i][1], pa[i][2], pa[i][3], bl[j], bh[j]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[st]));
    consumer_sync();  // P and red_max are rewritten by the next tile
  }

  // ---- finish: l per head across the column tiles, O / l, lse
  float l0 = lpart[0], l1 = lpart[1];
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, off);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, off);
  }
  if (t == 0) {
    red_l[mt][nt][g] = l0;
    red_l[mt][nt][g + 8] = l1;
    if (nt == 0) {
      red_max[mt][0][g] = mref[0];  // the reference maxima, shared with the output warps
      red_max[mt][0][g + 8] = mref[1];
    }
  }
  consumer_sync();
  if (timed_out && lane == 0) atomicOr(a.status, kErrWaitTimeout);
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int hr = 16 * i + g + 8 * hh;
      const int head = h0 + hr;
      float lt = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) lt += red_l[i][k][g + 8 * hh];
      const float inv = lt > 0.f ? a.out_scale / lt : 0.f;
      if (head < a.H) {
        // n-tile j, columns 2t, 2t+1 of the fragment <-> head_dim 32 w + 4 (2t..2t+1) + j
        uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + ((int64_t)b * a.H + head) * kDv + 32 * warp;
        uint32_t pk[4];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          pk[2 * c] = pack_bf16x2(o[i][0][2 * hh + c] * inv, o[i][1][2 * hh + c] * inv);
          pk[2 * c + 1] = pack_bf16x2(o[i][2][2 * hh + c] * inv, o[i][3][2 * hh + c] * inv);
        }
        *reinterpret_cast<uint2*>(dst + 4 * (2 * t)) = make_uint2(pk[0], pk[1]);
        *reinterpret_cast<uint2*>(dst + 4 * (2 * t + 1)) = make_uint2(pk[2], pk[3]);
        if (a.lse && warp == 0 && t == 0)
          a.lse[(int64_t)b * a.H + head] =
              lt > 0.f ? (red_max[i][0][g + 8 * hh] + __log2f(lt)) * kLn2 : -INFINITY;
      }
    }
}

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
  if (num_heads % 16 != 0 || num_heads > 128)
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
    if (cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
      return check_cuda("mla_decode set smem attribute");
    attr_set = true;
  }
  if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), s) != cudaSuccess)
    return check_cuda("mla_decode status reset");
  dim3 grid(batch, (num_heads + kHeads - 1) / kHeads);
  mla_decode_kernel<<<grid, kThreads, kSmemBytes, s>>>(a);
  return check_cuda("mla_decode launch");
}

}  // extern "C"
