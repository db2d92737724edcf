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
// the pair splits the score contraction instead of repeating it: CTA r
// contracts latent columns 256 r .. 256 r + 255 (Q held in tensor memory as
// the A operand) and rope columns 512 + 32 r .. 512 + 32 r + 31 (Q in shared
// memory).  The partial score tiles cross between the pair through
// distributed shared memory, one bulk copy per tile, as 16-bit fixed point
// over the row's range in the tile (an fp32 row minimum, a power-of-two step
// with range / step <= 65535, one u16 code per token: error <= range / 65535
// in log2 units).  Each CTA adds its own exact fp32 partial to the peer's
// decoded one, runs the online softmax over the sum and multiplies its P tile
// into its own output columns; each half is normalised by its own running sum.
//
// Per 32-token tile, with four tiles in flight (scores and P in tensor
// memory, the widened latent tile in shared memory):
//   producer warp   resolves the cache rows of 1024 list positions at a time
//                   (top-k entry -> block table, cached in shared memory ->
//                   row) into a double-buffered shared table;
//   loader warps    (8 rows of every tile each) gather this CTA's 288 bytes of
//                   each row with 16-byte asynchronous copies five tiles
//                   ahead (the rate of random row gathers grows with the
//                   number of issuing warps), then widen their rows to f16
//                   (exact) in the 128-byte-swizzled layout the MMA reads,
//                   K-major for the scores and MN-major for the output;
//   MMA thread      S[128 x 32] = Q . C^T (18 K steps), and two tiles later
//                   O += P . C[:, own 256] (2 K steps, N = 256);
//   sender warps    read S, encode it and copy it to the peer;
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
constexpr int kAhead = 5;             // tiles a loader warp gathers ahead of the one it widens
constexpr int kXDepth = 3;            // exchange buffers per direction
constexpr int kLatCols = 256;         // latent columns one CTA contracts (and outputs)
constexpr int kRopeCols = 32;         // rope columns one CTA contracts
constexpr int kRowCopy = kLatCols + kRopeCols;  // 288 staged bytes per token row
constexpr int kRowChunks = kRowCopy / 16;        // 18; chunk c of staged row r sits at (c + r) % 18
constexpr int kLoadRows = kTok / 4;               // rows per loader warp
constexpr int kSlotBytes = kLoadRows * kRowCopy;   // one loader warp's rows of one tile, e4m3
constexpr int kStageBytes = 4 * (kAhead + 1) * kSlotBytes;  // all loader warps' staging
constexpr int kAtomBytes = kTok * 128;           // [32 tokens][64 f16 columns], 128-byte swizzle
constexpr int kCBufBytes = 5 * kAtomBytes;       // 4 latent atoms + the rope atom
constexpr int kQRopeBytes = kRows * 128;         // [128 heads][64 rope columns] f16
constexpr int kXCodes = kRows * kTok * 2;        // exchanged partial scores: [128][32] u16 codes
constexpr int kXBytes = kXCodes + kRows * 4 + kRows;  // + [128] fp32 row minima + [128] step exponents
constexpr int kRowTab = 1024;                    // list positions per half of the row table
constexpr int kRowTabTiles = kRowTab / kTok;
constexpr int kBtCache = 2048;                   // block-table entries cached in shared memory

constexpr int kOffQRope = 0;
constexpr int kOffC = kOffQRope + kQRopeBytes;
constexpr int kOffStage = kOffC + kBufs * kCBufBytes;
constexpr int kOffSend = kOffStage + kStageBytes;
constexpr int kOffRecv = kOffSend + kXDepth * kXBytes;
constexpr int kOffRows = kOffRecv + kXDepth * kXBytes;
constexpr int kOffBt = kOffRows + 2 * kRowTab * 4;
constexpr int kOffBars = kOffBt + kBtCache * 4;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;        // 256 columns: this CTA's output columns, fp32
constexpr uint32_t kTmemS = 256;      // 4 x 32 columns: scores, then P (f16 pairs) in the first 16
constexpr uint32_t kTmemQ = 384;      // 128 columns: this CTA's 256 latent Q columns as f16 pairs

constexpr int kLoadWarp0 = 0;         // warps 0-3
constexpr int kSoftWarp0 = 4;         // warps 4-7: TMEM lane quadrants 0-3
constexpr int kSendWarp0 = 8;         // warps 8-11: TMEM lane quadrants 0-3
constexpr int kProdWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kAckWarp = 14;
constexpr int kThreads = 15 * 32;
constexpr int kPvLag = 2;             // the MMA thread issues O += P(j - 2) C(j - 2) after S(j)

constexpr uint32_t kIdescQK = tc::idesc_f16(kRows, kTok, false);
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
  int topk_n, B, H, P, max_pages;
  int64_t num_pages;
  float score_scale;  // ckv_scale * softmax_scale * log2(e)
  float out_scale;    // ckv_scale
};

struct __align__(8) Bars {
  uint64_t rows_ready[2], rows_free[2];  // the two halves of the row table
  uint64_t cfull[kBufs], sfull[kBufs], pfull[kBufs], pvdone[kBufs];
  uint64_t sent[kBufs];      // the sender warps have read the scores of a tile
  uint64_t qready;
  uint64_t xfull[kXDepth];   // the peer's partial scores of a tile have landed
  uint64_t xack[kXDepth];    // the peer has read a tile this CTA sent
  uint64_t rdone[kXDepth];   // this CTA's softmax warps have read a received tile
  uint32_t cmask[kBufs];  // bit i: token row i of the tile takes part (byte w from loader warp w)
  uint8_t vmask[4][kAhead + 1];  // loader warp w: which of its rows of a staged tile take part
  uint32_t tmem_base;
};
constexpr size_t kSmemBytes = (size_t)kOffBars + sizeof(Bars) + 1024;  // + alignment of the base to 1024
static_assert(kSmemBytes <= 232448, "shared memory over the per-CTA limit");

// 16-byte global -> shared copy through L2 only; completion is tracked per
// thread by commit groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most kAhead of this thread's committed groups are still landing.
__device__ __forceinline__ void cp_async_wait_ahead() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kAhead) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) { return pack_f16x2(bf16_lo(v), bf16_hi(v)); }

// Shared memory of this CTA -> shared memory of a peer CTA, completion
// counted in bytes on the peer's mbarrier.
__device__ __forceinline__ void bulk_to_peer(uint32_t dst_cluster, uint32_t src, uint32_t bytes, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(src), "r"(bytes), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ uint4 lds128_u32(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr) : "memory");
  return r;
}

// The four sender warps only.
__device__ __forceinline__ void sender_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// Byte offset of 16-byte unit c (0..3) of row t in an exchange buffer
// ([128][64 bytes], rows paired per 128-byte line): conflict-free for eight
// consecutive rows.
__device__ __forceinline__ uint32_t xunit(int t, int c) { return t * 64 + 16 * (c ^ ((t >> 1) & 3)); }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) mla_decode_kernel(const MlaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars& bs = *reinterpret_cast<Bars*>(smem + kOffBars);

  const uint32_t rank = tc::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int b = blockIdx.x >> 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int L = a.context_lens[b];
  if (L < 0) L = 0;
  if (L > a.max_pages * a.P) L = a.max_pages * a.P;
  const int n = a.topk ? a.topk_n : L;
  const int ntiles = (n + kTok - 1) / kTok;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bs.rows_ready[i]), 1);
      mbar_init(smem_u32(&bs.rows_free[i]), 4);
    }
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(smem_u32(&bs.cfull[i]), 4);
      mbar_init(smem_u32(&bs.sfull[i]), 1);
      mbar_init(smem_u32(&bs.pfull[i]), 4);
      mbar_init(smem_u32(&bs.pvdone[i]), 1);
      mbar_init(smem_u32(&bs.sent[i]), 4);
    }
    mbar_init(smem_u32(&bs.qready), 4);
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
  const uint32_t tmem = bs.tmem_base;
  bool to = false;  // this thread gave up a wait

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    // Row table half c % 2 <- list positions 1024 c .. 1024 c + 1023: top-k
    // entry -> page -> cache row (-1: padding, past the list, or rejected).
    const int64_t tbase = (int64_t)b * a.topk_n;
    const int32_t* bt = a.block_tables + (int64_t)b * a.max_pages;
    int32_t* bt_s = reinterpret_cast<int32_t*>(smem + kOffBt);
    const int npages = (L + a.P - 1) / a.P;
    const int ncached = npages < kBtCache ? npages : kBtCache;
#pragma unroll 1
    for (int i0 = 0; i0 < ncached; i0 += 32 * 16) {
      int v[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const int i = i0 + lane + 32 * m;
        v[m] = i < ncached ? bt[i] : 0;
      }
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const int i = i0 + lane + 32 * m;
        if (i < ncached) bt_s[i] = v[m];
      }
    }
    __syncwarp();
    const int nchunks = (n + kRowTab - 1) / kRowTab;
    for (int c = 0; c < nchunks; ++c) {
      if (c >= 2 && !to) to = !mbar_wait(smem_u32(&bs.rows_free[c & 1]), ((c - 2) >> 1) & 1);
      int32_t* rowtab = reinterpret_cast<int32_t*>(smem + kOffRows) + (c & 1) * kRowTab;
#pragma unroll 1
      for (int half = 0; half < kRowTab / 1024; ++half) {
        const int p0 = c * kRowTab + 32 * 32 * half + lane;
        int tok[32];
#pragma unroll
        for (int m = 0; m < 32; ++m) {
          const int p = p0 + 32 * m;
          tok[m] = p < n ? (a.topk ? a.topk[tbase + p] : p) : -1;
        }
#pragma unroll
        for (int m = 0; m < 32; ++m) {
          int32_t row = -1;
          const int tk = tok[m];
          if (tk >= L) {
            if (a.topk) atomicOr(a.status, kErrBadTopk);
          } else if (tk >= 0) {
            const int pi = tk / a.P;
            const int pg = pi < kBtCache ? bt_s[pi] : bt[pi];
            if (pg < 0 || (int64_t)pg >= a.num_pages)
              atomicOr(a.status, kErrBadPage);
            else
              row = pg * a.P + (tk - pi * a.P);
          }
          rowtab[32 * 32 * half + lane + 32 * m] = row;
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.rows_ready[c & 1]));
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      if (!to) to = !mbar_wait(smem_u32(&bs.qready), 0);
      tc::fence_after_sync();
      const uint32_t cbase0 = smem_u32(smem + kOffC), qrope = smem_u32(smem + kOffQRope);
      for (int j = 0; j < ntiles + kPvLag; ++j) {
        if (j < ntiles) {  // S(j) = Q . C(j)^T
          const int cb = j % kBufs;
          if (!to) to = !mbar_wait(smem_u32(&bs.cfull[cb]), (j / kBufs) & 1);
          tc::fence_after_sync();
          const uint32_t cbuf = cbase0 + cb * kCBufBytes;
          const uint32_t d = tmem + kTmemS + kTok * cb;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            tc::mma_ts(d, tmem + kTmemQ + 8 * k, tc::desc_sw128(cbuf + (k >> 2) * kAtomBytes + 32 * (k & 3), 16, 1024),
                       kIdescQK, k > 0);
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint32_t koff = 32 * (2 * rank + k);
            tc::mma_ss(d, tc::desc_sw128(qrope + koff, 16, 1024),
                       tc::desc_sw128(cbuf + 4 * kAtomBytes + koff, 16, 1024), kIdescQK, 1);
          }
          tc::mma_commit(smem_u32(&bs.sfull[cb]));
        }
        if (j >= kPvLag) {  // O += P(pj) . C(pj)[:, own columns]
          const int pj = j - kPvLag, pb = pj % kBufs;
          if (!to) to = !mbar_wait(smem_u32(&bs.pfull[pb]), (pj / kBufs) & 1);
          tc::fence_after_sync();
          const uint32_t cbuf = cbase0 + pb * kCBufBytes;
#pragma unroll
          for (int k = 0; k < kTok / 16; ++k)
            tc::mma_ts(tmem + kTmemO, tmem + kTmemS + kTok * pb + 8 * k,
                       tc::desc_sw128(cbuf + 2048 * k, kAtomBytes, 1024), kIdescPV, (pj > 0 || k > 0));
          tc::mma_commit(smem_u32(&bs.pvdone[pb]));
        }
      }
      // no MMA may still be running when the tensor memory is freed
      if (ntiles > 0 && !to)
        to = !mbar_wait(smem_u32(&bs.pvdone[(ntiles - 1) % kBufs]), ((ntiles - 1) / kBufs) & 1);
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
  } else if (warp < kLoadWarp0 + 4) {
    // --------------------------------------------------------- loader warps
    // Warp w owns token rows 8 w .. 8 w + 7 of every tile: it gathers them
    // (e4m3, 18 chunks of 16 bytes per row: 16 latent, 2 rope) into staging
    // slot (tile % 6) five tiles ahead, then widens them to f16 in the
    // swizzled atoms of latent buffer tile % 4.
    const int w = warp - kLoadWarp0;
    const uint8_t* src_lat = a.ckv + kLatCols * rank;
    const uint8_t* src_rope = a.ckv + kDv + kRopeCols * rank;
    uint8_t* stage = smem + kOffStage + w * (kAhead + 1) * kSlotBytes;
    const int32_t* rowtab0 = reinterpret_cast<const int32_t*>(smem + kOffRows);
    auto issue = [&](int jj) {  // gather this warp's rows of tile jj (nothing past the list)
      if (jj < ntiles) {
        const int c = jj / kRowTabTiles;
        if (jj % kRowTabTiles == 0 && !to) to = !mbar_wait(smem_u32(&bs.rows_ready[c & 1]), (c >> 1) & 1);
        const int32_t* rt = rowtab0 + (c & 1) * kRowTab + kTok * (jj % kRowTabTiles) + kLoadRows * w;
        const uint32_t sdst = smem_u32(stage + (jj % (kAhead + 1)) * kSlotBytes);
#pragma unroll
        for (int k = 0; k < (kLoadRows * kRowChunks + 31) / 32; ++k) {
          const int i = lane + 32 * k;
          if (i < kLoadRows * kRowChunks) {
            const int r = i / kRowChunks, ch = i - r * kRowChunks;
            const int32_t row = rt[r];
            const int u = ch + r < kRowChunks ? ch + r : ch + r - kRowChunks;  // rotated: no bank conflicts
            if (row >= 0)
              cp_async16(sdst + r * kRowCopy + 16 * u,
                         (ch < 16 ? src_lat + 16 * ch : src_rope + 16 * (ch - 16)) + (int64_t)row * kDqk);
          }
        }
        const uint32_t vm = __ballot_sync(0xFFFFFFFFu, lane < kLoadRows && rt[lane < kLoadRows ? lane : 0] >= 0);
        if (lane == 0) bs.vmask[w][jj % (kAhead + 1)] = (uint8_t)vm;
        __syncwarp();
        const bool last_of_chunk = (jj % kRowTabTiles == kRowTabTiles - 1) || jj == ntiles - 1;
        if (last_of_chunk && lane == 0) tc::mbar_arrive_local(smem_u32(&bs.rows_free[c & 1]));
      }
      cp_async_commit();  // one group per tile, empty past the list
    };
    for (int jj = 0; jj < kAhead; ++jj) issue(jj);
    // widening: lane l takes row l % 8, chunks l / 8 + 4 m
    const int wr = lane & 7, wc0 = lane >> 3;
    const uint32_t swz = (kLoadRows * w + wr) & 7;
    for (int j = 0; j < ntiles; ++j) {
      const int cb = j % kBufs;
      issue(j + kAhead);
      cp_async_wait_ahead();  // this lane's copies of tile j have landed
      __syncwarp();           // ... and every lane's
      if (j >= kBufs && !to) to = !mbar_wait(smem_u32(&bs.pvdone[cb]), ((j - kBufs) / kBufs) & 1);
      const uint32_t bits = bs.vmask[w][j % (kAhead + 1)];
      const bool valid = (bits >> wr) & 1;
      const uint8_t* src = stage + (j % (kAhead + 1)) * kSlotBytes + wr * kRowCopy;
      uint8_t* cbuf = smem + kOffC + cb * kCBufBytes + (kLoadRows * w + wr) * 128;
#pragma unroll
      for (int m = 0; m < 5; ++m) {
        const int ch = wc0 + 4 * m;
        if (ch < kRowChunks) {
          uint4 v = make_uint4(0, 0, 0, 0);
          const int u = ch + wr < kRowChunks ? ch + wr : ch + wr - kRowChunks;
          if (valid) v = lds128(src + 16 * u);
          uint4 o0, o1;
          e4m3x4_to_f16x2x2(v.x, o0.x, o0.y);
          e4m3x4_to_f16x2x2(v.y, o0.z, o0.w);
          e4m3x4_to_f16x2x2(v.z, o1.x, o1.y);
          e4m3x4_to_f16x2x2(v.w, o1.z, o1.w);
          const int atom = ch < 16 ? (ch >> 2) : 4;
          const uint32_t unit = ch < 16 ? 2 * (ch & 3) : 4 * rank + 2 * (ch - 16);
          uint8_t* dst = cbuf + atom * kAtomBytes;
          *reinterpret_cast<uint4*>(dst + 16 * (unit ^ swz)) = o0;
          *reinterpret_cast<uint4*>(dst + 16 * ((unit + 1) ^ swz)) = o1;
        }
      }
      fence_proxy_async_smem();  // generic writes -> visible to the tensor core
      __syncwarp();
      if (lane == 0) {
        reinterpret_cast<uint8_t*>(&bs.cmask[cb])[w] = (uint8_t)bits;
        tc::mbar_arrive_local(smem_u32(&bs.cfull[cb]));
      }
    }
    cp_async_wait_all();  // nothing may still be landing when the CTA retires
  } else if (warp >= kSendWarp0) {
    // --------------------------------------------------------- sender warps
    // Tile j: this CTA's partial scores (log2 units) -> 16-bit fixed point in
    // send buffer j % 3 -> one bulk copy into the peer's receive buffer.
    const int t = threadIdx.x - kSendWarp0 * 32;  // head row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const float sc = a.score_scale;
    const uint32_t send0 = smem_u32(smem + kOffSend);
    const uint32_t peer_recv0 = tc::mapa(smem_u32(smem + kOffRecv), peer);
    for (int j = 0; j < ntiles; ++j) {
      const int sb = j % kBufs, xb = j % kXDepth;
      if (!to) to = !mbar_wait(smem_u32(&bs.sfull[sb]), (j / kBufs) & 1);
      // the copy of tile j - 3 out of this buffer has landed and been read
      if (j >= kXDepth && !to) to = !tc::mbar_wait_cluster(smem_u32(&bs.xack[xb]), ((j - kXDepth) / kXDepth) & 1);
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
      float lo = x[0], hi = x[0];
#pragma unroll
      for (int i = 1; i < 32; ++i) {
        lo = fminf(lo, x[i]);
        hi = fmaxf(hi, x[i]);
      }
      // step = 2^(e - 127), the smallest power of two with (hi - lo) / step <= 65535
      const uint32_t rb = __float_as_uint((hi - lo) * (1.f / 65535.f));
      uint32_t e = ((rb >> 23) & 0xFFu) + ((rb & 0x7FFFFFu) != 0u);
      e = e < 1u ? 1u : (e > 253u ? 253u : e);
      const float inv = __uint_as_float((254u - e) << 23);  // 1 / step, exact
      const uint32_t buf = send0 + xb * kXBytes;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t q0 = min(__float2uint_rn((x[8 * c + 2 * k] - lo) * inv), 65535u);
          const uint32_t q1 = min(__float2uint_rn((x[8 * c + 2 * k + 1] - lo) * inv), 65535u);
          w[k] = q0 | (q1 << 16);
        }
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(buf + xunit(t, c)), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3])
                     : "memory");
      }
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(buf + kXCodes + 4 * t), "f"(lo) : "memory");
      asm volatile("st.shared.u8 [%0], %1;" ::"r"(buf + kXCodes + 4 * kRows + t), "r"(e) : "memory");
      fence_proxy_async_smem();
      sender_sync();
      if (t == 0) {
        mbar_arrive_expect_tx(smem_u32(&bs.xfull[xb]), kXBytes);  // the peer's tile j, into recv buffer xb
        bulk_to_peer(peer_recv0 + xb * kXBytes, buf, kXBytes, tc::mapa(smem_u32(&bs.xfull[xb]), peer));
      }
    }
  } else {
    // ------------------------------------------------------- softmax warps
    const int t = threadIdx.x - kSoftWarp0 * 32;  // head row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    {  // Q: this CTA's latent columns into tensor memory, the rope into shared memory
      const bool have = t < a.H;
      const __nv_bfloat16* qrow = a.q + ((int64_t)b * a.H + (have ? t : 0)) * kDqk;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint4 x = make_uint4(0, 0, 0, 0);
          if (have) x = ldg_nc(qrow + kLatCols * rank + 64 * c + 8 * u);
          v[4 * u + 0] = bf16x2_to_f16x2(x.x);
          v[4 * u + 1] = bf16x2_to_f16x2(x.y);
          v[4 * u + 2] = bf16x2_to_f16x2(x.z);
          v[4 * u + 3] = bf16x2_to_f16x2(x.w);
        }
        tc::tmem_st32(tl + kTmemQ + 32 * c, v);
      }
      uint8_t* qr = smem + kOffQRope + t * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint4 x = make_uint4(0, 0, 0, 0);
        if (have) x = ldg_nc(qrow + kDv + 8 * u);
        const uint4 y = make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                                   bf16x2_to_f16x2(x.w));
        *reinterpret_cast<uint4*>(qr + 16 * (u ^ (t & 7))) = y;
      }
      tc::tmem_st_wait();
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.qready));
    }

    const float sc = a.score_scale;
    const uint32_t recv0 = smem_u32(smem + kOffRecv);
    float mref = -INFINITY, l = 0.f;
    for (int j = 0; j < ntiles; ++j) {
      const int sb = j % kBufs, xb = j % kXDepth;
      if (!to) to = !mbar_wait(smem_u32(&bs.sfull[sb]), (j / kBufs) & 1);
      if (!to) to = !mbar_wait(smem_u32(&bs.cfull[sb]), (j / kBufs) & 1);
      if (!to) to = !tc::mbar_wait_cluster(smem_u32(&bs.xfull[xb]), (j / kXDepth) & 1);
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
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(plo) : "r"(theirs + kXCodes + 4 * t) : "memory");
        asm volatile("ld.shared.u8 %0, [%1];" : "=r"(pe) : "r"(theirs + kXCodes + 4 * kRows + t) : "memory");
        const float pstep = __uint_as_float(pe << 23);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 hq = lds128_u32(theirs + xunit(t, c));
          const uint32_t wq[4] = {hq.x, hq.y, hq.z, hq.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float p0 = fmaf(__uint2float_rn(wq[k] & 0xFFFFu), pstep, plo);
            const float p1 = fmaf(__uint2float_rn(wq[k] >> 16), pstep, plo);
            s[8 * c + 2 * k] = fmaf(__uint_as_float(v[8 * c + 2 * k]), sc, p0);
            s[8 * c + 2 * k + 1] = fmaf(__uint_as_float(v[8 * c + 2 * k + 1]), sc, p1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.rdone[xb]));  // the ack warp frees it at the peer

      // ---- mask, tile maximum, lazy reference update
      const uint32_t mask = bs.cmask[sb];
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = ((mask >> i) & 1) ? s[i] : -INFINITY;
        mx = fmaxf(mx, s[i]);
      }
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

  if (to) atomicOr(a.status, kErrWaitTimeout);
  tc::fence_before_sync();
  tc::cluster_sync();  // the peer no longer touches this CTA's shared memory
  tc::fence_after_sync();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
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
  mla_decode_kernel<<<dim3(2 * batch), kThreads, kSmemBytes, s>>>(a);
  return check_cuda("mla_decode launch");
}

}  // extern "C"
