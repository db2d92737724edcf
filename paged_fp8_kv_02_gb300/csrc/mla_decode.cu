// mla_decode.cu -- MLA absorbed-latent decode over one shared e4m3 latent row
// per token, optionally restricted to a top-k token list, on the fifth-
// generation tensor cores (tcgen05, accumulators in tensor memory).
//
// kLLM article (快手万擎大模型推理成本和性能优化实践), §5.1.1: DSA selects the
// top-k historical tokens that take part in attention and MLA stores a
// compressed per-token latent cKV; §5.1.2: that latent is shared by all heads
// (it cannot be split by head the way GQA KV heads can).  Absorbed reading: the
// whole Dqk = 576-wide row is the key, its first 512 entries are the value.
//
// Per request a cluster of two CTAs.  The fp32 output O[128 heads][512] alone
// fills one SM's tensor memory, so CTA r keeps O[:, 256 r .. 256 r + 255] and
// the pair splits the score contraction instead of repeating it: CTA 0
// contracts latent columns 0 .. 255, CTA 1 latent columns 256 .. 511 and the
// 64 rope columns (Q's latent part held in tensor memory as the A operand,
// the rope part in shared memory, both f16; a row whose largest |q| over the
// CTA's columns lies outside [2^-4, 2^15] is first scaled by a power of two,
// undone on that CTA's partial scores), so each CTA reads one contiguous span of
// every row (256 or 320 bytes).  The partial score tiles cross between the
// pair through distributed shared memory (asynchronous remote stores that
// count their bytes on the receiver's mbarrier) as 16-bit fixed point
// over the row's range in the tile (an fp32 row minimum, a power-of-two step
// with range / step <= 65535, one u16 code per token: error <= range / 65535
// in log2 units).  Each CTA adds its own exact fp32 partial to the peer's
// decoded one, runs the online softmax over the sum and multiplies its P tile
// into its own output columns; each half is normalised by its own running sum.
//
// Per 32-token tile, with four tiles in flight (scores and P in tensor
// memory, the widened latent tiles in shared memory, two tiles per buffer so
// that the scores of a tile pair come from one N = 64 MMA sequence):
//   producer warp   resolves the cache rows of 2048 list positions at a time
//                   (top-k entry -> block table, cached in shared memory ->
//                   row) into a shared table and gathers this CTA's span of
//                   each row with TMA four-row gathers (tile::gather4) into a
//                   5-stage e4m3 ring;
//   converter warps widen the tile to f16 (exact) in the 128-byte-swizzled
//                   layout the MMA reads, K-major for the scores and MN-major
//                   for the output product;
//   MMA thread      S[128 x 64] = Q . C^T for a tile pair (16 or 20 K steps) and
//                   O += P . C[:, own 256] (2 K steps, N = 256), each issued
//                   as soon as its inputs are ready;
//   sender warps    read S, encode it and store it into the peer's receive
//                   buffer;
//   softmax warps   (one TMEM lane per head) add the peer's partial, take the
//                   exp2 online softmax with a reference maximum that moves
//                   only when a score exceeds it by more than 2^8 (then O is
//                   rescaled in tensor memory) and store P as f16 pairs over
//                   the score columns, where the MMA reads it as its A operand;
//   ack warp        tells the peer when a received tile has been read.
// Every wait is bounded; a wait that gives up sets PFKV_DEVERR_WAIT_TIMEOUT
// and the CTA still runs to its end, so the pair always meets at the final
// cluster barrier and frees its tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "pfkv_internal.h"
#include "pfkv_ptx.cuh"
#include "pfkv_tc.cuh"

namespace pfkv {
namespace {

constexpr int kDqk = 576, kDv = 512;
constexpr int kRows = 128;            // MMA rows: query heads, zero-padded
constexpr int kTok = 32;              // tokens per tile
constexpr int kBufs = 4;              // tiles in flight: score/P buffers and widened latent tiles
constexpr int kStages = 5;            // e4m3 staging ring
constexpr int kXDepth = 3;            // exchange buffers per direction
constexpr int kLatCols = 256;         // latent columns one CTA contracts (and outputs)
constexpr int kSpan0 = 256, kSpan1 = 320;  // bytes of each row CTA 0 / CTA 1 reads
constexpr int kStageBytes = kTok * kSpan1;
constexpr int kAtomBytes = 2 * kTok * 128;       // [64 tokens: a tile pair][64 f16 columns], 128-byte swizzle
constexpr int kCBufBytes = 5 * kAtomBytes;       // 4 latent atoms + the rope atom, for a tile pair
constexpr int kPairs = kBufs / 2;                // pair buffers
constexpr int kQRopeBytes = kRows * 128;         // [128 heads][64 rope columns] f16
constexpr int kXCodes = kRows * kTok * 2;        // exchanged partial scores: [128][32] u16 codes
constexpr int kXMeta = kRows * 8;                // per row: fp32 minimum, u32 step exponent
constexpr int kXBytes = kXCodes + kXMeta;
constexpr int kChunkTiles = 8;                   // tiles per chunk of resolved rows
constexpr int kChunkPos = kChunkTiles * kTok;    // 256 list positions
constexpr int kRowSlots = 8;                     // chunks of resolved rows in flight
constexpr int kRowTab = kRowSlots * kChunkPos;   // 2048 entries

constexpr int kOffQRope = 0;
constexpr int kOffC = kOffQRope + kQRopeBytes;
constexpr int kOffStage = kOffC + kPairs * kCBufBytes;
constexpr int kOffRecv = kOffStage + kStages * kStageBytes;
constexpr int kOffRows = kOffRecv + kXDepth * kXBytes;
constexpr int kOffBars = kOffRows + kRowTab * 4;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;        // 256 columns: this CTA's output columns, fp32
constexpr uint32_t kTmemS = 256;      // 4 x 32 columns: scores, then P (f16 pairs) in the first 16
constexpr uint32_t kTmemQ = 384;      // 128 columns: this CTA's 256 latent Q columns as f16 pairs

constexpr int kConvWarp0 = 0;         // warps 0-3
constexpr int kSoftWarp0 = 4;         // warps 4-7: TMEM lane quadrants 0-3
constexpr int kSendWarp0 = 8;         // warps 8-11: TMEM lane quadrants 0-3
constexpr int kProdWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kAckWarp = 14;
constexpr int kResWarp = 15;          // resolves list positions to cache rows ahead of the producer
constexpr int kThreads = 16 * 32;

constexpr uint32_t kIdescQK = tc::idesc_f16(kRows, 2 * kTok, false);
constexpr uint32_t kIdescPV = tc::idesc_f16(kRows, kLatCols, true);

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;

struct MlaArgs {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const uint8_t* ckv;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* topk;
  float* lse;
  int32_t* status;
  float* part_o;      // split calls: raw O of every (request, split) [B * nsplit][H][512] fp32
  float2* part_ml;    // split calls: (reference, running sum) [B * nsplit][2 halves][H]
  int nsplit;         // clusters per request (list positions split into nsplit runs)
  int chunk_pos;      // list positions per split (a multiple of 32)
  int topk_n, B, H, P, max_pages;
  int p_shift;        // log2(P) when P is a power of two, else -1
  int64_t num_pages;
  float score_scale;  // ckv_scale * softmax_scale * log2(e)
  float out_scale;    // ckv_scale
};

struct __align__(8) Bars {
  uint64_t stage_full[kStages], stage_empty[kStages];
  uint64_t cfull[kBufs], sfull[kBufs], pfull[kBufs], pvdone[kBufs];
  uint64_t sent[kBufs];      // the sender warps have read the scores of a tile
  uint64_t qready;
  float qinv[kRows];         // 1 / the power-of-two Q scale of each head row (this CTA's columns)
  uint64_t xfull[kXDepth];   // the peer's partial scores of a tile have landed
  uint64_t xack[kXDepth];    // the peer has read a tile this CTA sent
  uint64_t rdone[kXDepth];   // this CTA's softmax warps have read a received tile
  uint64_t rows_full[kRowSlots], rows_empty[kRowSlots];  // a chunk of resolved rows written / issued
  uint32_t stage_mask[kStages], cmask[kBufs];  // bit i: token row i of the tile takes part
  uint32_t tmem_base;
};
constexpr size_t kSmemBytes = (size_t)kOffBars + sizeof(Bars) + 1024;  // + alignment of the base to 1024
static_assert(kSmemBytes <= 232448, "shared memory over the per-CTA limit");

// Four rows (y0..y3) of a 2D tensor map, columns x .. x + box - 1, into
// consecutive box-wide rows of shared memory; completion counted in bytes on
// the mbarrier.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int y0, int y1, int y2,
                                            int y3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
      : "memory");
}

// bf16 pair times a power of two -> f16 pair
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v, float s) {
  return pack_f16x2(bf16_lo(v) * s, bf16_hi(v) * s);
}

// Remote stores into a peer CTA's shared memory whose bytes are counted on
// the peer's mbarrier when they land (no separate arrival needed).
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void st_async_v2(uint32_t addr, uint32_t a, uint32_t b, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "r"(a), "r"(b), "r"(bar)
               : "memory");
}

__device__ __forceinline__ uint4 lds128_u32(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr) : "memory");
  return r;
}

// Maximum / minimum of 32 values as a tree (short dependency chains).
__device__ __forceinline__ float tree_max32(const float (&x)[32]) {
  float m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = fmaxf(x[2 * i], x[2 * i + 1]);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  return m[0];
}
__device__ __forceinline__ float tree_min32(const float (&x)[32]) {
  float m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = fminf(x[2 * i], x[2 * i + 1]);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fminf(m[i], m[i + w]);
  return m[0];
}
// u16 codes <-> floats through the 2^23 bias: for 0 <= v <= 65535 the fp32
// sum v + 2^23 holds round(v) in its low mantissa bits, and the float with
// exponent 2^23 and low bits q equals 2^23 + q exactly.
constexpr float kTwo23 = 8388608.f;
__device__ __forceinline__ uint32_t biased_code(float v) { return __float_as_uint(v + kTwo23); }
__device__ __forceinline__ float code_lo(uint32_t w) { return __uint_as_float(prmt(w, 0x4B000000u, 0x7410)) - kTwo23; }
__device__ __forceinline__ float code_hi(uint32_t w) { return __uint_as_float(prmt(w, 0x4B000000u, 0x7432)) - kTwo23; }

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Byte offset of 16-byte unit c (0..3) of row t in an exchange buffer
// ([128][64 bytes], rows paired per 128-byte line): conflict-free for eight
// consecutive rows.
__device__ __forceinline__ uint32_t xunit(int t, int c) { return t * 64 + 16 * (c ^ ((t >> 1) & 3)); }

// tm0 / tm1: the cache as [rows][288 u16], boxes of 128 / 160 columns (CTA 0 / CTA 1).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                      const MlaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars& bs = *reinterpret_cast<Bars*>(smem + kOffBars);

  const uint32_t rank = tc::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cid = blockIdx.x >> 1;           // cluster: (request, split of its list)
  const int b = cid / a.nsplit, split = cid - b * a.nsplit;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int L = a.context_lens[b];
  if (L < 0) L = 0;
  if (L > a.max_pages * a.P) L = a.max_pages * a.P;
  // this cluster's run of list positions: p0 .. p0 + n - 1
  const int p0 = split * a.chunk_pos;
  const int n_all = a.topk ? a.topk_n : L;
  const int n = max(0, min(n_all - p0, a.chunk_pos));
  const int ntiles = (n + kTok - 1) / kTok;

  // This CTA's span of the request's query rows (128-byte lines 4 rank ..
  // 4 rank + 3 of each 1152-byte row, plus line 8, the rope, for rank 1) into
  // L2 now, so that the conversion below reads them from L2 while the
  // barriers, tensor memory and the first gathers are set up.
  {
    const int lines = rank ? 5 : 4;
    const char* q0 = reinterpret_cast<const char*>(a.q + (int64_t)b * a.H * kDqk) + 512 * rank;
    for (int i = threadIdx.x; i < a.H * lines; i += kThreads) {
      const int row = i / lines, ln = i - row * lines;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(q0 + (int64_t)row * (2 * kDqk) + 128 * ln));
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bs.stage_full[s]), 1);
      mbar_init(smem_u32(&bs.stage_empty[s]), 4);
    }
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(smem_u32(&bs.cfull[i]), 4);
      mbar_init(smem_u32(&bs.sfull[i]), 1);
      mbar_init(smem_u32(&bs.pfull[i]), 4);
      mbar_init(smem_u32(&bs.pvdone[i]), 1);
      mbar_init(smem_u32(&bs.sent[i]), 4);
    }
    mbar_init(smem_u32(&bs.qready), 4);
    for (int i = 0; i < kRowSlots; ++i) {
      mbar_init(smem_u32(&bs.rows_full[i]), 1);
      mbar_init(smem_u32(&bs.rows_empty[i]), 1);
    }
    for (int i = 0; i < kXDepth; ++i) {
      mbar_init(smem_u32(&bs.xfull[i]), 1);
      mbar_init(smem_u32(&bs.xack[i]), 1);
      mbar_init(smem_u32(&bs.rdone[i]), 4);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(smem_u32(&bs.tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  tc::cluster_sync();  // both CTAs' barriers initialised before any remote arrival
  tc::fence_after_sync();
  grid_launch_dependents();  // the merge of a split call may be scheduled as CTAs retire
  const uint32_t tmem = bs.tmem_base;
  bool to = false;  // this thread gave up a wait

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    // Rows come from the resolver warp in chunks of kChunkTiles tiles.
    const int32_t* rowtab = reinterpret_cast<const int32_t*>(smem + kOffRows);
    const CUtensorMap* tm = rank ? &tm1 : &tm0;
    const int span = rank ? kSpan1 : kSpan0;
    const int x0 = rank ? kLatCols / 2 : 0;  // first u16 column of this CTA's span
    for (int j = 0; j < ntiles; ++j) {
      const int chunk = j / kChunkTiles, slot = chunk % kRowSlots;
      if (j % kChunkTiles == 0 && !to)
        to = !__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bs.rows_full[slot]), (chunk / kRowSlots) & 1));
      if (to) break;
      const int st = j % kStages;
      if (j >= kStages && !to) to = !mbar_wait(smem_u32(&bs.stage_empty[st]), ((j / kStages) - 1) & 1);
      const int32_t* rt = rowtab + slot * kChunkPos + kTok * (j % kChunkTiles);
      const uint32_t mask = __ballot_sync(0xFFFFFFFFu, rt[lane] >= 0);
      const uint32_t full = smem_u32(&bs.stage_full[st]);
      if (lane == 0) {
        bs.stage_mask[st] = mask;
        mbar_arrive_expect_tx(full, (uint32_t)(kTok * span));
      }
      __syncwarp();
      if (lane < kTok / 4) {  // rows that take no part fetch row 0 and are zeroed when widened
        const int r = 4 * lane;
        const int y0 = rt[r] >= 0 ? rt[r] : 0, y1 = rt[r + 1] >= 0 ? rt[r + 1] : 0;
        const int y2 = rt[r + 2] >= 0 ? rt[r + 2] : 0, y3 = rt[r + 3] >= 0 ? rt[r + 3] : 0;
        tma_gather4(smem_u32(smem + kOffStage + st * kStageBytes + r * span), tm, x0, y0, y1, y2, y3, full);
      }
      __syncwarp();
      // the chunk's rows have all been issued: the resolver may reuse its slot
      if (lane == 0 && (j % kChunkTiles == kChunkTiles - 1 || j == ntiles - 1))
        tc::mbar_arrive_local(smem_u32(&bs.rows_empty[slot]));
    }
    // no copy may still be landing when the CTA retires
    for (int j = ntiles > kStages ? ntiles - kStages : 0; j < ntiles; ++j)
      if (!to) to = !mbar_wait(smem_u32(&bs.stage_full[j % kStages]), (j / kStages) & 1);
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // Issues O += P(j) . C(j)[:, own columns] as soon as P(j) is stored (first:
    // it frees a widened tile buffer), and S = Q . C^T for a tile pair as soon
    // as both tiles are widened and their score columns are free; the scores
    // run up to four tiles ahead.
    if (lane == 0) {
      if (!to) to = !mbar_wait(smem_u32(&bs.qready), 0);
      tc::fence_after_sync();
      const uint32_t cbase0 = smem_u32(smem + kOffC);
      const uint64_t qdesc = tc::desc_sw128(smem_u32(smem + kOffQRope), 16, 1024);
      int qn = 0, pn = 0;  // next tile for the scores (even: a pair) / for the output
      long long idle_since = clock64();
      while (pn < ntiles && !to) {
        bool issued = false;
        if (pn < qn && mbar_test_wait(smem_u32(&bs.pfull[pn % kBufs]), (pn / kBufs) & 1)) {
          tc::fence_after_sync();
          const uint64_t vdesc =
              tc::desc_sw128(cbase0 + ((pn / 2) % kPairs) * kCBufBytes + (pn & 1) * kTok * 128, kAtomBytes, 1024);
#pragma unroll
          for (int k = 0; k < kTok / 16; ++k)
            tc::mma_ts(tmem + kTmemO, tmem + kTmemS + kTok * (pn % kBufs) + 8 * k, vdesc + (uint64_t)((2048 * k) >> 4),
                       kIdescPV, (pn > 0 || k > 0));
          tc::mma_commit(smem_u32(&bs.pvdone[pn % kBufs]));
          ++pn;
          issued = true;
        }
        // the pair's score columns held P(qn - 4) and P(qn - 3): both products issued
        if (qn < ntiles && pn >= qn - 2 && mbar_test_wait(smem_u32(&bs.cfull[qn % kBufs]), (qn / kBufs) & 1) &&
            (qn + 1 >= ntiles || mbar_test_wait(smem_u32(&bs.cfull[(qn + 1) % kBufs]), ((qn + 1) / kBufs) & 1))) {
          tc::fence_after_sync();
          // descriptors built once; K steps add constant offsets to the address field
          const uint64_t bdesc = tc::desc_sw128(cbase0 + ((qn / 2) % kPairs) * kCBufBytes, 16, 1024);
          const uint32_t d = tmem + kTmemS + kTok * (qn % kBufs);
#pragma unroll
          for (int k = 0; k < 16; ++k)
            tc::mma_ts(d, tmem + kTmemQ + 8 * k, bdesc + (uint64_t)(((k >> 2) * kAtomBytes + 32 * (k & 3)) >> 4),
                       kIdescQK, k > 0);
          if (rank) {  // the 64 rope columns
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_ss(d, qdesc + (uint64_t)((32 * k) >> 4), bdesc + (uint64_t)((4 * kAtomBytes + 32 * k) >> 4),
                         kIdescQK, 1);
          }
          tc::mma_commit(smem_u32(&bs.sfull[qn % kBufs]));
          if (qn + 1 < ntiles) tc::mma_commit(smem_u32(&bs.sfull[(qn + 1) % kBufs]));
          qn += 2;
          issued = true;
        }
        if (issued) {
          idle_since = clock64();
        } else {
          __nanosleep(32);  // leave issue slots to the warps sharing this scheduler
          if (clock64() - idle_since > kWaitLimitCycles) to = true;
        }
      }
      // no MMA may still be running when the tensor memory is freed
      if (ntiles > 0 && pn > 0 && !mbar_wait(smem_u32(&bs.pvdone[(pn - 1) % kBufs]), ((pn - 1) / kBufs) & 1))
        to = true;
    }
    __syncwarp();
  } else if (warp == kAckWarp) {
    // ------------------------------------------------------------- ack warp
    if (lane == 0) {
      for (int j = 0; j < ntiles; ++j) {
        const int xb = j % kXDepth;
        if (!to) to = !mbar_wait(smem_u32(&bs.rdone[xb]), (j / kXDepth) & 1);
        tc::mbar_arrive_remote(tc::mapa(smem_u32(&bs.xack[xb]), peer));
      }
    }
    __syncwarp();
  } else if (warp < kConvWarp0 + 4) {
    // ---------------------------------------------------------- converters
    // 16-byte chunk i of the staged tile (row i / nch, chunk i % nch; chunks
    // 0-15 latent, 16-19 rope) -> e4m3 -> f16 -> the swizzled atoms.
    // Consecutive threads read consecutive chunks of a row; the offsets are
    // the same for every tile.
    const int nch = rank ? kSpan1 / 16 : kSpan0 / 16;
    const int span = rank ? kSpan1 : kSpan0;
    constexpr int kChunksPerThread = kSpan1 / 16 * kTok / 128;  // 5
    int src_off[kChunksPerThread], dst_off[kChunksPerThread], crow[kChunksPerThread];
#pragma unroll
    for (int m = 0; m < kChunksPerThread; ++m) {
      const int i = threadIdx.x - kConvWarp0 * 32 + 128 * m;
      const int row = i / nch, ch = i - (i / nch) * nch;
      const int atom = ch < 16 ? (ch >> 2) : 4;
      const uint32_t unit = ch < 16 ? 2 * (ch & 3) : 2 * (ch - 16);
      crow[m] = i < nch * kTok ? row : -1;
      src_off[m] = row * span + 16 * ch;
      dst_off[m] = atom * kAtomBytes + row * 128 + 16 * (unit ^ (row & 7));  // unit + 1: ^ 16
    }
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % kStages, cb = j % kBufs;
      if (!to) to = !mbar_wait(smem_u32(&bs.stage_full[st]), (j / kStages) & 1);
      if (j >= kBufs && !to) to = !mbar_wait(smem_u32(&bs.pvdone[cb]), ((j - kBufs) / kBufs) & 1);
      const uint32_t mask = bs.stage_mask[st];
      const uint8_t* stage = smem + kOffStage + st * kStageBytes;
      uint8_t* cbuf = smem + kOffC + ((j / 2) % kPairs) * kCBufBytes + (j & 1) * kTok * 128;
      // every load before the first store: the compiler cannot move a load
      // above a store through another pointer into shared memory
      uint4 v[kChunksPerThread];
#pragma unroll
      for (int m = 0; m < kChunksPerThread; ++m) {
        v[m] = make_uint4(0, 0, 0, 0);
        if (crow[m] >= 0 && ((mask >> crow[m]) & 1)) v[m] = lds128(stage + src_off[m]);
      }
#pragma unroll
      for (int m = 0; m < kChunksPerThread; ++m) {
        if (crow[m] >= 0) {
          uint4 o0, o1;
          e4m3x4_to_f16x2x2(v[m].x, o0.x, o0.y);
          e4m3x4_to_f16x2x2(v[m].y, o0.z, o0.w);
          e4m3x4_to_f16x2x2(v[m].z, o1.x, o1.y);
          e4m3x4_to_f16x2x2(v[m].w, o1.z, o1.w);
          // units u and u + 1 (u even) differ in bit 0, so their swizzled
          // positions differ by exactly 16 bytes
          *reinterpret_cast<uint4*>(cbuf + dst_off[m]) = o0;
          *reinterpret_cast<uint4*>(cbuf + (dst_off[m] ^ 16)) = o1;
        }
      }
      fence_proxy_async_smem();  // generic writes -> visible to the tensor core
      __syncwarp();
      if (lane == 0) {
        if (warp == kConvWarp0) bs.cmask[cb] = mask;
        tc::mbar_arrive_local(smem_u32(&bs.stage_empty[st]));
        tc::mbar_arrive_local(smem_u32(&bs.cfull[cb]));
      }
    }
  } else if (warp == kResWarp) {
    // ------------------------------------------------------------ resolver
    // List position p -> top-k entry -> page -> cache row (-1: padding, past
    // the list, or rejected), a chunk of 256 positions at a time (eight per
    // lane, loads in flight together), up to kRowSlots chunks ahead of the
    // producer.
    const int64_t tbase = (int64_t)b * a.topk_n;
    const int32_t* bt = a.block_tables + (int64_t)b * a.max_pages;
    int32_t* rowtab = reinterpret_cast<int32_t*>(smem + kOffRows);
    const int nchunks = (ntiles + kChunkTiles - 1) / kChunkTiles;
    for (int c = 0; c < nchunks && !to; ++c) {
      const int slot = c % kRowSlots;
      if (c >= kRowSlots &&
          !__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&bs.rows_empty[slot]), ((c / kRowSlots) - 1) & 1))) {
        to = true;
        break;
      }
      int tok[8], pg[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int p = c * kChunkPos + lane + 32 * m;
        tok[m] = p < n ? (a.topk ? a.topk[tbase + p0 + p] : p0 + p) : -1;
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int tk = tok[m];
        pg[m] = (tk >= 0 && tk < L) ? bt[a.p_shift >= 0 ? tk >> a.p_shift : tk / a.P] : -1;
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        int32_t row = -1;
        const int tk = tok[m];
        if (tk >= L) {
          if (a.topk) atomicOr(a.status, kErrBadTopk);
        } else if (tk >= 0) {
          const int pi = a.p_shift >= 0 ? tk >> a.p_shift : tk / a.P;
          if (pg[m] < 0 || (int64_t)pg[m] >= a.num_pages)
            atomicOr(a.status, kErrBadPage);
          else
            row = pg[m] * a.P + (tk - pi * a.P);
        }
        rowtab[slot * kChunkPos + lane + 32 * m] = row;
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.rows_full[slot]));
    }
  } else if (warp >= kSendWarp0) {
    // --------------------------------------------------------- sender warps
    // Tile j: this CTA's partial scores (log2 units) -> 16-bit fixed point,
    // stored straight into the peer's receive buffer j % 3.
    const int t = threadIdx.x - kSendWarp0 * 32;  // head row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t peer_recv0 = tc::mapa(smem_u32(smem + kOffRecv), peer);
    if (!to) to = !mbar_wait(smem_u32(&bs.qready), 0);  // the rows' Q scales are written
    const float sc = a.score_scale * bs.qinv[t];
    for (int j = 0; j < ntiles; ++j) {
      const int sb = j % kBufs, xb = j % kXDepth;
      if (!to) to = !mbar_wait(smem_u32(&bs.sfull[sb]), (j / kBufs) & 1);
      tc::fence_after_sync();
      float x[32];
      {
        uint32_t v[32];
        tc::tmem_ld32(tl + kTmemS + kTok * sb, v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]) * sc;
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.sent[sb]));  // the softmax may overwrite S with P
      // the peer has read tile j - 3 out of the buffer this tile goes to
      if (j >= kXDepth && !to) to = !tc::mbar_wait_cluster(smem_u32(&bs.xack[xb]), ((j - kXDepth) / kXDepth) & 1);
      const float lo = tree_min32(x), hi = tree_max32(x);
      // step = 2^(e - 127), the smallest power of two with (hi - lo) / step <= 65535
      const uint32_t rb = __float_as_uint((hi - lo) * (1.f / 65535.f));
      uint32_t e = ((rb >> 23) & 0xFFu) + ((rb & 0x7FFFFFu) != 0u);
      e = e < 1u ? 1u : (e > 253u ? 253u : e);
      const float inv = __uint_as_float((254u - e) << 23);  // 1 / step, exact
      const uint32_t dst = peer_recv0 + xb * kXBytes;
      const uint32_t rbar = tc::mapa(smem_u32(&bs.xfull[xb]), peer);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // (x - lo) * inv is exact and <= (hi - lo) * inv <= 65535: no clamp needed
          const uint32_t q0 = biased_code((x[8 * c + 2 * k] - lo) * inv);
          const uint32_t q1 = biased_code((x[8 * c + 2 * k + 1] - lo) * inv);
          w[k] = prmt(q0, q1, 0x5410);
        }
        st_async_v4(dst + xunit(t, c), w[0], w[1], w[2], w[3], rbar);
      }
      st_async_v2(dst + kXCodes + 8 * t, __float_as_uint(lo), e, rbar);
    }
  } else {
    // ------------------------------------------------------- softmax warps
    const int t = threadIdx.x - kSoftWarp0 * 32;  // head row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    // Q: this CTA's latent columns into tensor memory, the rope into shared
    // memory, as f16.  A row whose largest |q| (over these columns) lies in
    // [2^-4, 2^15] converts as it is: it fits f16 and every value at least
    // 2^-10 of the largest is an exact f16 normal.  Any other row is
    // converted again after a power-of-two scale qs taking its largest |q|
    // into (2^14, 2^15]; 1 / qs joins this CTA's score scale (here and in
    // the sender warps).
    float qinv_row = 1.f;
    {
      const bool have = t < a.H;
      const __nv_bfloat16* qrow = a.q + ((int64_t)b * a.H + (have ? t : 0)) * kDqk;
      uint8_t* qr = smem + kOffQRope + t * 128;
      float amax = 0.f;
      auto convert = [&](float qs) {
        // two chunks of 64 columns per round: sixteen 16-byte loads in flight
#pragma unroll 1
        for (int c0 = 0; c0 < 4; c0 += 2) {
          uint4 xs[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            xs[u] = make_uint4(0, 0, 0, 0);
            if (have) xs[u] = ldg_nc(qrow + kLatCols * rank + 64 * c0 + 8 * u);
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t v[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 x = xs[8 * cc + u];
              const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
                v[4 * u + k] = bf16x2_to_f16x2(w[k], qs);
              }
            }
            tc::tmem_st32(tl + kTmemQ + 32 * (c0 + cc), v);
          }
        }
#pragma unroll
        for (int u = 0; u < 8 * (int)rank; ++u) {
          uint4 x = make_uint4(0, 0, 0, 0);
          if (have) x = ldg_nc(qrow + kDv + 8 * u);
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
          const uint4 y = make_uint4(bf16x2_to_f16x2(x.x, qs), bf16x2_to_f16x2(x.y, qs),
                                     bf16x2_to_f16x2(x.z, qs), bf16x2_to_f16x2(x.w, qs));
          *reinterpret_cast<uint4*>(qr + 16 * (u ^ (t & 7))) = y;
        }
      };
      convert(1.f);
      const bool rescale = amax > 32768.f || (amax > 0.f && amax < 0.0625f);
      if (__any_sync(0xFFFFFFFFu, rescale)) {  // the whole warp: tensor-memory stores are warp-wide
        const float qs = rescale ? pow2_scale(32768.f, amax) : 1.f;
        qinv_row = 1.f / qs;  // exact: qs is a power of two
        tc::tmem_st_wait();   // the first conversion's stores complete before they are overwritten
        convert(qs);
      }
      bs.qinv[t] = qinv_row;
      tc::tmem_st_wait();
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.qready));
    }

    const float sc = a.score_scale * qinv_row;
    const uint32_t recv0 = smem_u32(smem + kOffRecv);
    float mref = -INFINITY, l = 0.f;
    // Receive buffer xb expects the peer's tile j only once its tile j - 3 has
    // been taken, so the expectation never lands in an earlier phase.
    if (t == 0)
      for (int j = 0; j < kXDepth && j < ntiles; ++j) mbar_arrive_expect_tx(smem_u32(&bs.xfull[j]), kXBytes);
    for (int j = 0; j < ntiles; ++j) {
      const int sb = j % kBufs, xb = j % kXDepth;
      if (!to) to = !mbar_wait(smem_u32(&bs.sfull[sb]), (j / kBufs) & 1);
      if (!to) to = !mbar_wait(smem_u32(&bs.cfull[sb]), (j / kBufs) & 1);
      if (!to) to = !tc::mbar_wait_cluster(smem_u32(&bs.xfull[xb]), (j / kXDepth) & 1);
      if (t == 0 && j + kXDepth < ntiles) mbar_arrive_expect_tx(smem_u32(&bs.xfull[xb]), kXBytes);
      tc::fence_after_sync();
      // ---- s = own exact partial + the peer's decoded partial
      float s[32];
      {
        uint32_t v[32];
        tc::tmem_ld32(tl + kTmemS + kTok * sb, v);
        tc::tmem_ld_wait();
        const uint32_t theirs = recv0 + xb * kXBytes;
        float plo;
        uint32_t pe;
        uint32_t plo_bits;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(plo_bits), "=r"(pe) : "r"(theirs + kXCodes + 8 * t) : "memory");
        plo = __uint_as_float(plo_bits);
        const float pstep = __uint_as_float(pe << 23);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 hq = lds128_u32(theirs + xunit(t, c));
          const uint32_t wq[4] = {hq.x, hq.y, hq.z, hq.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float p0 = fmaf(code_lo(wq[k]), pstep, plo);
            const float p1 = fmaf(code_hi(wq[k]), pstep, plo);
            s[8 * c + 2 * k] = fmaf(__uint_as_float(v[8 * c + 2 * k]), sc, p0);
            s[8 * c + 2 * k + 1] = fmaf(__uint_as_float(v[8 * c + 2 * k + 1]), sc, p1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.rdone[xb]));  // the ack warp frees it at the peer

      // ---- mask, tile maximum, lazy reference update
      const uint32_t mask = bs.cmask[sb];
      if (mask != 0xFFFFFFFFu) {
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = ((mask >> i) & 1) ? s[i] : -INFINITY;
      }
      const float mx = tree_max32(s);
      const bool grow = mx > mref + kRescaleLog2;
      float alpha = 1.f;
      if (grow) {
        alpha = fast_exp2(mref - mx);  // 0 when there was no reference yet
        mref = mx;
        l *= alpha;
      }
      if (j > 0 && __any_sync(0xFFFFFFFFu, grow)) {  // O *= alpha once PV(j-1) has landed
        if (!to) to = !mbar_wait(smem_u32(&bs.pvdone[(j - 1) % kBufs]), ((j - 1) / kBufs) & 1);
        tc::fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < kLatCols / 32; ++c) {
          uint32_t v[32];
          tc::tmem_ld32(tl + kTmemO + 32 * c, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tc::tmem_st32(tl + kTmemO + 32 * c, v);
        }
      }
      // ---- P = 2^(s - ref) as f16 pairs over the score columns
      const float moff = mref == -INFINITY ? 0.f : mref;
      uint32_t pk[16];
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = fast_exp2(s[2 * i] - moff), p1 = fast_exp2(s[2 * i + 1] - moff);
        lsum += p0 + p1;
        pk[i] = pack_f16x2(p0, p1);
      }
      l += lsum;
      if (!to) to = !mbar_wait(smem_u32(&bs.sent[sb]), (j / kBufs) & 1);  // the sender has read S(j)
      tc::fence_after_sync();
      tc::tmem_st16(tl + kTmemS + kTok * sb, pk);
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.pfull[sb]));
    }

    // ---- epilogue: O / l -> bf16, this CTA's 256 columns; lse from rank 0
    if (ntiles > 0 && !to)
      to = !mbar_wait(smem_u32(&bs.pvdone[(ntiles - 1) % kBufs]), ((ntiles - 1) / kBufs) & 1);
    tc::fence_after_sync();
    if (a.nsplit > 1) {
      // A run of a split list: the raw accumulator, reference and sum go to
      // the workspace; mla_merge_kernel folds the runs by log-sum-exp.  Each
      // 32-column chunk of this warp's 32 rows goes through shared memory (the
      // widened-tile buffers, idle once the last output product is done) so
      // that every store instruction writes whole 128-byte runs of 4 rows.
      float* stg = reinterpret_cast<float*>(smem + kOffC) + (warp - kSoftWarp0) * (32 * 33);
      const int64_t u = (int64_t)b * a.nsplit + split;
#pragma unroll 1
      for (int c = 0; c < kLatCols / 32; ++c) {
        uint32_t v[32];
        if (ntiles > 0) {
          tc::tmem_ld32(tl + kTmemO + 32 * c, v);
          tc::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) stg[lane * 33 + i] = __uint_as_float(v[i]);
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = 4 * k + (lane >> 3), c4 = 4 * (lane & 7);
          const int row = 32 * (warp - kSoftWarp0) + r;  // head
          const float* sp = stg + r * 33 + c4;
          if (row < a.H)
            *reinterpret_cast<float4*>(a.part_o + (u * a.H + row) * kDv + kLatCols * rank + 32 * c + c4) =
                make_float4(sp[0], sp[1], sp[2], sp[3]);
        }
        __syncwarp();  // the staging rows are rewritten by the next chunk
      }
      if (t < a.H) a.part_ml[(u * 2 + rank) * a.H + t] = make_float2(l > 0.f ? mref : -INFINITY, l);
    } else {
      const float inv = l > 0.f ? a.out_scale / l : 0.f;
      uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + ((int64_t)b * a.H + t) * kDv + kLatCols * rank;
#pragma unroll 1
      for (int c = 0; c < kLatCols / 32; ++c) {
        uint32_t v[32];
        if (ntiles > 0) {
          tc::tmem_ld32(tl + kTmemO + 32 * c, v);
          tc::tmem_ld_wait();
        }
        if (t < a.H) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = l > 0.f ? pack_bf16x2(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv) : 0u;
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (rank == 0 && a.lse && t < a.H)
        a.lse[(int64_t)b * a.H + t] = l > 0.f ? (mref + __log2f(l)) * kLn2 : -INFINITY;
    }
  }

  if (to) atomicOr(a.status, kErrWaitTimeout);
  tc::fence_before_sync();
  tc::cluster_sync();  // the peer no longer touches this CTA's shared memory
  tc::fence_after_sync();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
}

// Folds the splits of each (request, head) row: with m_s the reference (log2
// units) and l_s the running sum of split s for this half of the columns,
// M = max_s m_s, out = ckv_scale * sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s
// (kLLM article §5.2.2: blockwise (m, l, O) states combine to full attention).
// One warp per row; lane i takes columns 4i .. 4i + 3 of each 128-column block.
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(kMergeWarps * 32) mla_merge_kernel(const MlaArgs a) {
  grid_dependency_wait();  // every run's state is written and visible
  const int row = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.B * a.H) return;
  const int b = row / a.H, hh = row - b * a.H;
  float lse_val = -INFINITY;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float M = -INFINITY;
    for (int s = 0; s < a.nsplit; ++s)
      M = fmaxf(M, a.part_ml[(((int64_t)b * a.nsplit + s) * 2 + half) * a.H + hh].x);
    float Lsum = 0.f;
    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int s = 0; s < a.nsplit; ++s) {
      const int64_t u = (int64_t)b * a.nsplit + s;
      const float2 ml = a.part_ml[(u * 2 + half) * a.H + hh];
      if (!(ml.y > 0.f)) continue;
      const float w = exp2f(ml.x - M);
      Lsum += w * ml.y;
      const float* src = a.part_o + (u * a.H + hh) * kDv + kLatCols * half;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float4 o = *reinterpret_cast<const float4*>(src + 128 * k + 4 * lane);
        acc[k].x += w * o.x;
        acc[k].y += w * o.y;
        acc[k].z += w * o.z;
        acc[k].w += w * o.w;
      }
    }
    const float inv = Lsum > 0.f ? a.out_scale / Lsum : 0.f;
    uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + (int64_t)row * kDv + kLatCols * half;
#pragma unroll
    for (int k = 0; k < 2; ++k)
      *reinterpret_cast<uint2*>(dst + 128 * k + 4 * lane) =
          make_uint2(pack_bf16x2(acc[k].x * inv, acc[k].y * inv), pack_bf16x2(acc[k].z * inv, acc[k].w * inv));
    if (half == 0) lse_val = Lsum > 0.f ? (M + __log2f(Lsum)) * kLn2 : -INFINITY;
  }
  if (a.lse && lane == 0) a.lse[row] = lse_val;
}

// Clusters per request: enough to fill the GPU's SM pairs (one cluster of two
// CTAs per pair) when the batch alone does not, each split taking at least
// kMinSplitTiles tiles of the list.
constexpr int kMinSplitTiles = 8;
constexpr size_t kWsHead = 256;  // status word
size_t split_bytes(int num_heads) { return (size_t)num_heads * (kDv * sizeof(float) + 2 * sizeof(float2)); }
int max_splits(int batch, int64_t list_len) {
  if (batch <= 0) return 1;
  const int pairs = device_sm_count() / 2;
  int ns = pairs / batch;
  const int64_t tiles = (list_len + kTok - 1) / kTok;
  const int64_t by_len = tiles / kMinSplitTiles;
  if (ns > by_len) ns = (int)by_len;
  return ns < 1 ? 1 : ns;
}

}  // namespace
}  // namespace pfkv

extern "C" {

size_t pfkv_mla_decode_workspace_size(int batch, int num_heads, int d_latent, int topk) {
  (void)d_latent;
  using namespace pfkv;
  if (batch <= 0 || num_heads <= 0) return kWsHead;
  // topk <= 0 (every token attended): the split count is bounded by the SM pairs alone
  const int ns = max_splits(batch, topk > 0 ? topk : ((int64_t)1 << 30));
  if (ns <= 1) return kWsHead;
  return kWsHead + (size_t)batch * ns * split_bytes(num_heads);
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
  if (num_heads % 16 != 0 || num_heads > kRows)
    return fail(PFKV_ERR_UNSUPPORTED, "mla_decode: num_heads must be a multiple of 16, <= 128");
  if (page_size % 16 != 0)
    return fail(PFKV_ERR_UNSUPPORTED, "mla_decode: page_size must be a multiple of 16");
  if (!isfinite(ckv_scale) || !isfinite(softmax_scale) || !(softmax_scale > 0.f))
    return fail(PFKV_ERR_INVALID_ARG, "mla_decode: scales must be finite");
  if (num_pages > (int64_t)INT32_MAX / page_size)
    return fail(PFKV_ERR_UNSUPPORTED, "mla_decode: more than 2^31 cache rows");
  if (batch == 0) return PFKV_OK;
  if (!out || !q || !ckv_cache || !block_tables || !context_lens || !workspace)
    return fail(PFKV_ERR_INVALID_ARG, "mla_decode: null pointer");
  if (workspace_bytes < 256) return fail(PFKV_ERR_WORKSPACE, "mla_decode: workspace too small");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(ckv_cache, 16) || !aligned(workspace, 256) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || (topk_idx && !aligned(topk_idx, 4)) ||
      (lse_out && !aligned(lse_out, 4)))
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
  a.p_shift = (page_size & (page_size - 1)) == 0 ? __builtin_ctz((unsigned)page_size) : -1;
  a.max_pages = max_pages_per_seq;
  a.num_pages = num_pages;
  a.score_scale = ckv_scale * softmax_scale * kLog2e;
  a.out_scale = ckv_scale;
  // split each request's list over several clusters when the batch leaves SM
  // pairs idle, as far as the workspace holds the partial states
  const int64_t list_len = topk_idx ? (int64_t)topk : (int64_t)max_pages_per_seq * page_size;
  int nsplit = max_splits(batch, list_len);
  while (nsplit > 1 && kWsHead + (size_t)batch * nsplit * split_bytes(num_heads) > workspace_bytes) --nsplit;
  const int64_t tiles = (list_len + kTok - 1) / kTok;
  a.nsplit = nsplit;
  a.chunk_pos = (int)(((tiles + nsplit - 1) / nsplit) * kTok);
  a.part_o = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kWsHead);
  a.part_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + kWsHead +
                                        (size_t)batch * nsplit * num_heads * kDv * sizeof(float));
  static std::atomic<uint64_t> smem_set{0};
  const int smem_rc = set_max_dynamic_smem(reinterpret_cast<const void*>(mla_decode_kernel), (int)kSmemBytes, smem_set,
                                       "mla_decode set smem attribute");
  if (smem_rc != PFKV_OK) return smem_rc;
  if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), s) != cudaSuccess)
    return check_cuda("mla_decode status reset");
  // The cache as [rows][288 u16]: CTA 0 reads u16 columns 0..127, CTA 1 128..287.
  const cuuint64_t dims[2] = {kDqk / 2, (cuuint64_t)num_pages * page_size};
  const cuuint64_t strides[1] = {kDqk};
  CUtensorMap tm0, tm1;
  const cuuint32_t box0[2] = {kSpan0 / 2, 1}, box1[2] = {kSpan1 / 2, 1};
  int rc = encode_tensor_map(&tm0, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(ckv_cache), dims, strides,
                             box0, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc == PFKV_OK)
    rc = encode_tensor_map(&tm1, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(ckv_cache), dims, strides,
                           box1, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != PFKV_OK) return rc;
  mla_decode_kernel<<<dim3(2 * batch * nsplit), kThreads, kSmemBytes, s>>>(tm0, tm1, a);
  if (nsplit > 1) {
    // a programmatic dependent: its launch overlaps the tail of the decode
    // kernel; it waits (griddepcontrol.wait) before reading the run states
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((batch * num_heads + kMergeWarps - 1) / kMergeWarps);
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(&cfg, mla_merge_kernel, a) != cudaSuccess) return check_cuda("mla_decode merge launch");
  }
  return check_cuda("mla_decode launch");
}

}  // extern "C"
