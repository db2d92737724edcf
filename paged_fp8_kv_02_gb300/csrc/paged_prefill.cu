// paged_prefill.cu -- attention of several new query tokens per request over
// the paged e4m3 cache, causal among the new tokens, on the fifth-generation
// tensor cores (tcgen05, operands in shared and tensor memory).
//
// Inference-engine scheduling explainer (推論エンジンの実践), section
// "チャンク分割と、その大きさの決め方": chunked prefill writes a prompt's KV chunk
// by chunk, and each chunk's tokens attend the cached prefix and each other;
// "Speculative Decoding" section: the target model checks the drafted
// positions in one parallel forward pass.  Both are this operation: request b
// has n_b query tokens at positions L_b - n_b .. L_b - 1, and query i attends
// keys 0 .. L_b - n_b + i.
//
// With several queries per KV head the step becomes a dense contraction, so
// the products run on tcgen05 with fp32 accumulation in tensor memory.  A row
// is one (query token, query head) pair of a KV head; a request's rows form
// blocks of 128 (128 / G query tokens per block).  Two kernels:
//   * prefillm_kernel, blocks of more than 64 rows (chunked prefill): one
//     128-row block per CTA over 128-token tiles; Q's two exact e4m3 parts in
//     tensor memory as the A operand of the score products (kind::f8f6f4,
//     straight on the K rows of the TMA stage); V widened to f16 for P.V
//     (kind::f16, P read from tensor memory); eight softmax warps, two per
//     lane quadrant, each taking half of a row's scores;
//   * prefillw_kernel, blocks of at most 64 rows (a few queries per request:
//     speculative verification): 128-token tiles with half-height (M = 64)
//     products, Q's parts in shared memory, the (request, KV head, tile) space
//     split evenly over one persistent CTA per SM.
// Both: K/V tiles gathered by TMA through the block table, boxes as tall as
// the page allows; lazy-reference exp2 online softmax (the reference moves
// only when a score exceeds it by more than 2^8; O in tensor memory is then
// rescaled); each Q row scaled by a power of two (largest |q| into
// (224, 448]) before the split, its 1 / scale joined to the score scale, so
// any finite bf16 query is accepted.  Pieces of one row's context computed
// apart (chunks of kv_split_tokens, or the even split's CTA boundaries) write
// fp32 partial states (m, l, o) that a merge kernel folds by the log-sum-exp
// rule (kLLM article, §5.2.2).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pfkv_internal.h"
#include "pfkv_ptx.cuh"
#include "pfkv_tc.cuh"

namespace pfkv {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;                    // rows of a work unit's block (one per MMA row)
constexpr int kTokN = 64;                     // granularity of kv_split_tokens and of unit tile counts
constexpr int kBoxTok = 16;                   // tokens per TMA box unless the page allows taller ones
constexpr int kBoxBytes = kBoxTok * kD;       // 2 KB
constexpr int kPartStride = 132;              // floats per row of a partial state: m, l, -, -, o[128]
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kTmemCols = 512;

struct PrefillArgs {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* q_start;
  float* lse;
  int32_t* status;
  float* partials;  // [units][kRows][kPartStride] when C > 1
  int B, Hq, Hkv, G, P, max_pages;
  int QB;           // row blocks per (request, KV head)
  int C;            // KV chunks per (request, KV head)
  int split;        // tokens per chunk
  int max_q_len, max_ctx;
  int64_t num_pages;
  float score_scale;  // k_scale * softmax_scale * log2(e)
  float out_scale;    // v_scale
  int box_tok;        // prefillw_kernel: tokens per TMA box (16, 32 or 64, dividing the page)
  int64_t* tile_start;  // prefillw_kernel: [B + 1] flattened start of each request's (KV head, tile) range
  int ncta;             // prefillw_kernel: CTAs sharing the flattened range
};

// Geometry of one (request, KV head, row block, chunk) unit, the same in both
// kernels.  Lengths are clamped to what the launch covers; the tile kernel
// reports clamping in the status word.
struct Unit {
  int b, kvh, qb, c;
  int L, n;          // clamped context length and query count
  int i0, i1;        // query tokens [i0, i1) of this block
  int rows;          // valid rows: (i1 - i0) * G
  int t_lo, t_hi;    // KV tokens [t_lo, t_hi) this unit reads (t_hi may be <= t_lo)
  int t_end_chunk;   // min(L, t_lo + split): the chunk's own end
  int ntiles;
  bool active;       // the unit exists (its block has queries and its chunk starts inside L)
};

__device__ __forceinline__ Unit unit_of(const PrefillArgs& a, int64_t u, bool report) {
  Unit x;
  x.qb = (int)(u % a.QB);
  int64_t r = u / a.QB;
  x.c = (int)(r % a.C);
  r /= a.C;
  x.kvh = (int)(r % a.Hkv);
  x.b = (int)(r / a.Hkv);
  const int L_raw = a.context_lens[x.b];
  const int n_raw = a.q_start[x.b + 1] - a.q_start[x.b];
  int cap = a.max_pages * a.P;
  if (a.max_ctx < cap) cap = a.max_ctx;
  int L = L_raw < 0 ? 0 : (L_raw > cap ? cap : L_raw);
  int ncap = L < a.max_q_len ? L : a.max_q_len;
  int n = n_raw < 0 ? 0 : (n_raw > ncap ? ncap : n_raw);
  if (report && (L != L_raw || n != n_raw)) atomicOr(a.status, kErrBadContext);
  x.L = L;
  x.n = n;
  const int tpb = kRows / a.G;
  x.i0 = x.qb * tpb;
  x.i1 = min(n, x.i0 + tpb);
  x.rows = (x.i1 - x.i0) * a.G;
  x.t_lo = x.c * a.split;
  x.active = x.i0 < n && x.t_lo < L;
  const int64_t chunk_end = (int64_t)x.t_lo + a.split;
  x.t_end_chunk = (int)(chunk_end < L ? chunk_end : L);
  const int qpos_max = L - n + x.i1 - 1;
  x.t_hi = min(x.t_end_chunk, qpos_max + 1);
  x.ntiles = x.active && x.t_hi > x.t_lo ? (x.t_hi - x.t_lo + kTokN - 1) / kTokN : 0;
  return x;
}

// Bounded wait taken by every lane of a warp, with one verdict for all lanes
// (so that a timeout never splits the warp).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity));
}

// 128-byte-swizzled offset of 16-byte chunk c of row r in a TMA box written
// with CU_TENSOR_MAP_SWIZZLE_128B (1024-byte aligned).
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// Offset of f16 unit u (elements 8u .. 8u+7, u < 16) of row r in a pair of
// 128-byte-swizzled K-major atoms [rows][64] (atom size atom_bytes).
__device__ __forceinline__ uint32_t atom_off(int r, int u, int atom_bytes) {
  return (uint32_t)((u >> 3) * atom_bytes + r * 128 + 16 * ((u & 7) ^ (r & 7)));
}

// ------------------------------------------ wide tiles for a few queries
// When every row block holds at most 64 rows (a few query tokens per request:
// speculative verification), prefillw_kernel uses 128-token tiles and
// half-height (M = 64) products, so that one score instruction covers 128
// tokens and each tile's fixed costs (waits, tensor-memory round trips) are
// spread over twice as many tokens.  The softmax reads the 16 rows of each
// warp with the 16-lane tensor-memory shape, so all 32 threads work (threads t
// and t ^ 2 share a row, each holding the columns of one parity).  So that a
// thread can pack its own P pairs, the contraction order of P.V swaps the
// middle two tokens of every group of four: P column pair (4r + 2e, 4r + 2e + 1)
// holds tokens (4r + e, 4r + e + 2), and row 4r + i of the widened V tile holds
// token 4r + (i with its two low bits swapped).  The score products read the
// e4m3 K rows straight from the TMA stage (kind::f8f6f4): each Q row is
// scaled by a power of two (its largest element into (224, 448]) and split
// into two e4m3 parts: a bf16 value has 8 significant bits and each part holds
// 4 (the remainder after rounding to the first is at most half its last unit),
// so the split is exact for every scaled element above 0.25 (checked over all
// bf16 values); smaller ones, below 1/896 of the row's largest, are off by at
// most half e4m3's subnormal step, 2^-10, under 2^-17 of the largest; so
// S = part 1 . K + part 2 . K, accumulated in fp32, and only V is
// widened to f16.  Each resource is released as soon as its last reader is done:
//   * P has tensor-memory columns of its own: a score buffer is free once the
//     softmax warps have read it, not once P.V has run;
//   * P is double-buffered: the softmax writes P(j) once P.V(j - 2) has read
//     that buffer, so P.V(j - 1) and the softmax of tile j overlap (O is
//     waited for only on the rare tiles whose reference moves);
//   * a stage is free once its K has been read by the score products and its
//     V widened; a widened V tile once its P.V product has run.
// tensor memory: two 128-column score buffers, O (128), two P buffers (64 each).
// shared memory: four 32 KB e4m3 stages, two 32 KB widened V tiles, Q's parts (16 KB).
constexpr int kWTok = 128;                      // tokens per tile
constexpr int kWStages = 4;
constexpr int kWStageBytes = 2 * kWTok * kD;    // K + V e4m3: 32 KB
constexpr int kWAtom = kWTok * 128;             // [128 tokens][64 f16]: 16 KB
constexpr int kWVBytes = 2 * kWAtom;            // widened V (2 atoms): 32 KB
constexpr int kWQPart = 64 * 128;               // one e4m3 part of Q: [64 rows][128 bytes], 8 KB
constexpr int kWBufs = 2;
constexpr int kWOffV = 0;
constexpr int kWOffStage = kWOffV + kWBufs * kWVBytes;
constexpr int kWOffQ = kWOffStage + kWStages * kWStageBytes;  // two parts
constexpr int kWOffQs = kWOffQ + 2 * kWQPart;                 // float[64]: each row's 1 / (Q scale)
constexpr int kWOffBars = kWOffQs + 64 * 4;
constexpr int kWSmemBytes = kWOffBars + 512 + 1024;
static_assert(kWSmemBytes <= 232448, "shared memory over the per-CTA limit");
constexpr uint32_t kWTmemS = 0, kWTmemO = kWBufs * kWTok, kWTmemP = kWTmemO + kD;
static_assert(kWTmemP + kWBufs * (kWTok / 2) <= kTmemCols, "tensor memory columns");
constexpr uint32_t kIdescQKW = tc::idesc_f16(64, kWTok, false);  // with kind::f8f6f4: e4m3 x e4m3
constexpr uint32_t kIdescPVW = tc::idesc_f16(64, kD, true);
constexpr int kWConvWarps = 4;
constexpr int kWProdWarp = 0, kWMmaWarp = 1, kWConvWarp0 = 2, kWSoftWarp0 = kWConvWarp0 + kWConvWarps,
              kWPvWarp = kWSoftWarp0 + 4, kWProdWarpV = kWPvWarp + 1;
constexpr int kWThreads = (kWProdWarpV + 1) * 32;
constexpr int kWChunks = kWTok * kD / 16 / (32 * kWConvWarps);  // 16-byte chunks of V per converter thread

struct BarsW {
  uint64_t stage_full[kWStages], stage_empty[kWStages];
  uint64_t vfull[kWBufs];                 // widened V of a tile written
  uint64_t sfull[kWBufs];                 // scores of a tile complete
  uint64_t sread[kWBufs];                 // the softmax warps have read a score buffer
  uint64_t pvdone[kWBufs];                // P.V of a tile complete (index: tile % 2)
  uint64_t pfull[kWBufs];                 // P of a tile written (index: tile % 2)
  uint64_t qready;                        // Q of the current segment written
  uint64_t qfree;                         // the previous segment's score products are done with Q
  uint64_t oread;                         // a segment's epilogue has read O
  uint32_t tmem_base;
};
static_assert(sizeof(BarsW) <= 512, "barrier block");
constexpr int kWRows = 64;  // rows of a block on this path (every block holds at most 64)

// Widening of a stage's V rows into f16 atoms, rows in the P.V contraction
// order, in two steps: load_v reads this thread's e4m3 chunks (rows at or past
// `valid` as zeros), so the stage can be released before the destination
// buffer is free; store_v converts and writes them.
__device__ __forceinline__ void load_v(const uint8_t* vstage, int ct, int valid, uint4 (&v)[kWChunks]) {
#pragma unroll
  for (int m = 0; m < kWChunks; ++m) {
    const int i = ct + 32 * kWConvWarps * m;  // row i / 8, 16-byte chunk i % 8
    const int row = i >> 3, c = i & 7;
    v[m] = make_uint4(0, 0, 0, 0);
    if (row < valid) v[m] = lds128(vstage + (row >> 4) * kBoxBytes + swz(row & 15, c));
  }
}
__device__ __forceinline__ void store_v(const uint4 (&v)[kWChunks], uint8_t* dst, int ct) {
#pragma unroll
  for (int m = 0; m < kWChunks; ++m) {
    const int i = ct + 32 * kWConvWarps * m;
    const int row = i >> 3, c = i & 7;
    uint4 o0, o1;
    e4m3x4_to_f16x2x2(v[m].x, o0.x, o0.y);
    e4m3x4_to_f16x2x2(v[m].y, o0.z, o0.w);
    e4m3x4_to_f16x2x2(v[m].z, o1.x, o1.y);
    e4m3x4_to_f16x2x2(v[m].w, o1.z, o1.w);
    const int drow = (row & ~3) | ((row & 1) << 1) | ((row >> 1) & 1);
    const uint32_t d = atom_off(drow, 2 * c, kWAtom);
    *reinterpret_cast<uint4*>(dst + d) = o0;
    *reinterpret_cast<uint4*>(dst + (d ^ 16)) = o1;
  }
}

// e4m3 code pair (byte 0 -> lo) -> two floats (exact).
__device__ __forceinline__ void e4m3x2_to_f32x2(uint16_t code, float& lo, float& hi) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(code));
  lo = __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
  hi = __half2float(__ushort_as_half((unsigned short)(h >> 16)));
}

// Clamped context length and query count of request b, as unit_of takes them.
__device__ __forceinline__ void clamped_ln(const PrefillArgs& a, int b, int& L, int& n, bool report) {
  const int L_raw = a.context_lens[b];
  const int n_raw = a.q_start[b + 1] - a.q_start[b];
  int cap = a.max_pages * a.P;
  if (a.max_ctx < cap) cap = a.max_ctx;
  L = L_raw < 0 ? 0 : (L_raw > cap ? cap : L_raw);
  const int ncap = L < a.max_q_len ? L : a.max_q_len;
  n = n_raw < 0 ? 0 : (n_raw > ncap ? ncap : n_raw);
  if (report && (L != L_raw || n != n_raw)) atomicOr(a.status, kErrBadContext);
}

// One CTA: tile_start[b] = sum over earlier requests of Hkv x their 128-token
// tiles (a request without queries has none); tile_start[B] = W.
__global__ void __launch_bounds__(1024) prefillw_plan_kernel(const PrefillArgs a) {
  __shared__ int64_t warp_sum[32];
  __shared__ int64_t carry;
  grid_launch_dependents();  // the tile kernel may start its prologue now
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int base = 0; base < a.B; base += 1024) {
    const int b = base + threadIdx.x;
    int64_t t = 0;
    if (b < a.B) {
      int L, n;
      clamped_ln(a, b, L, n, true);
      t = n > 0 ? (int64_t)((L + kWTok - 1) / kWTok) * a.Hkv : 0;
    }
    int64_t sc = t;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xFFFFFFFFu, sc, o);
      if (lane >= o) sc += y;
    }
    if (lane == 31) warp_sum[wid] = sc;
    __syncthreads();
    if (wid == 0) {
      int64_t w = warp_sum[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
        if (lane >= o) w += y;
      }
      warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int64_t before = carry + (wid > 0 ? warp_sum[wid - 1] : 0) + sc - t;
    if (b < a.B) a.tile_start[b] = before;
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_sum[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) a.tile_start[a.B] = carry;
}

// A CTA's run of tiles inside one (request, KV head): tiles [ta, tb) of its
// ceil(L / 128), as a unit (tokens [t_lo, t_hi), causal mask as usual).
struct Seg {
  Unit x;
  bool whole;    // the run is the pair's whole range: the output rows are written directly
  int64_t slot;  // otherwise its partial state's slot: CTA + b Hkv + kvh
};
__device__ __forceinline__ Seg seg_at(const PrefillArgs& a, int64_t f, int64_t f1) {
  // the last request whose range starts at or before f (it has tiles: f < W)
  int lo = 0, hi = a.B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.tile_start[mid] <= f) lo = mid;
    else hi = mid;
  }
  const int b = lo;
  const int64_t s0 = a.tile_start[b];
  const int per = (int)((a.tile_start[b + 1] - s0) / a.Hkv);  // tiles per KV head
  const int64_t off = f - s0;
  const int kvh = (int)(off / per), ta = (int)(off % per);
  const int64_t room = (int64_t)per - ta;
  const int tb = ta + (int)(f1 - f < room ? f1 - f : room);
  Seg sg;
  Unit& x = sg.x;
  int L, n;
  clamped_ln(a, b, L, n, false);
  x.b = b;
  x.kvh = kvh;
  x.qb = 0;
  x.c = 0;
  x.L = L;
  x.n = n;
  x.i0 = 0;
  x.i1 = n;
  x.rows = n * a.G;
  x.t_lo = ta * kWTok;
  x.t_hi = min(tb * kWTok, L);
  x.t_end_chunk = x.t_hi;
  x.ntiles = tb - ta;
  x.active = true;
  sg.whole = ta == 0 && tb == per;
  sg.slot = (int64_t)blockIdx.x + (int64_t)b * a.Hkv + kvh;
  return sg;
}

// Flattened and persistent: the (request, KV head, 128-token tile) space is
// laid out request by request (prefillw_plan_kernel writes where each
// request's range starts) and CTA i of N takes tiles [i W / N, (i + 1) W / N):
// every SM gets the same number of tiles whatever the mix of lengths.  A
// CTA's range is a few segments, one per (request, KV head) it touches; each
// warp role walks the same segments (a deterministic walk, no queue), and the
// producer streams the next segment's tiles while the current one drains.
// Every ring's phase follows the CTA's running tile count g.  A segment that
// covers its whole (request, KV head) writes the output rows; any other writes
// a partial state (m, l, o) to slot i + (b Hkv + kvh), distinct for every
// (CTA, pair) since a CTA's pairs are consecutive, and prefillw_merge_kernel
// folds them (kLLM article, §5.2.2).
// Per segment: the softmax warps write Q once the previous segment's score
// products are done (qfree) and signal qready; P.V of a segment's first tile
// overwrites O once the previous segment's epilogue has read it (oread).
__global__ void __launch_bounds__(kWThreads, 1)
    prefillw_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* const smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  BarsW& bs = *reinterpret_cast<BarsW*>(smem + kWOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(smem_u32(&bs.stage_full[s]), 2);  // the K and the V producer
      mbar_init(smem_u32(&bs.stage_empty[s]), kWConvWarps + 1);  // V read + the score products done
    }
    for (int k = 0; k < kWBufs; ++k) {
      mbar_init(smem_u32(&bs.vfull[k]), kWConvWarps);
      mbar_init(smem_u32(&bs.sfull[k]), 1);
      mbar_init(smem_u32(&bs.sread[k]), 4);
      mbar_init(smem_u32(&bs.pvdone[k]), 1);
      mbar_init(smem_u32(&bs.pfull[k]), 4);
    }
    mbar_init(smem_u32(&bs.qready), 4);
    mbar_init(smem_u32(&bs.qfree), 1);
    mbar_init(smem_u32(&bs.oread), 4);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == kWMmaWarp) {
    tc::tmem_alloc(smem_u32(&bs.tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bs.tmem_base;
  bool to = false;  // a bounded wait gave up

  grid_launch_dependents();  // the merge kernel may be scheduled as CTAs retire
  grid_dependency_wait();    // the plan's tile offsets are complete and visible
  const int64_t W = a.tile_start[a.B];
  const int64_t f0 = (int64_t)blockIdx.x * W / gridDim.x, f1 = ((int64_t)blockIdx.x + 1) * W / gridDim.x;

  if (warp == kWProdWarp || warp == kWProdWarpV) {
    // ------------------------------------------------------------ producers
    // warp kWProdWarp copies K, warp kWProdWarpV copies V, each arriving on
    // the stage with its own byte count (one warp issuing both measured slower)
    const bool isv = warp == kWProdWarpV;
    // A tile is nb = 128 / box_tok boxes per tensor, each inside one page
    // (tiles start at multiples of 64 tokens): with 64-token pages two 8 KB
    // copies instead of eight 2 KB ones, which measured faster.  A 64-row box
    // lands in shared memory exactly as four 16-row boxes would (the 128-byte
    // swizzle repeats every 8 rows).  Lane l holds the block-table entry of box
    // l % nb of tile (batch + l / nb), 32 / nb tiles per load, the next batch
    // loaded while this one is issued.
    const int btok = a.box_tok, nb = kWTok / btok, tpb = 32 / nb;
    int64_t g = 0;  // tiles issued by this CTA so far
    for (int64_t f = f0; f < f1 && !to;) {
      const Seg sg = seg_at(a, f, f1);
      const Unit& x = sg.x;
      const int ntiles = x.ntiles;
      const int32_t* bt = a.block_tables + (int64_t)x.b * a.max_pages;
      auto load_batch = [&](int j0) {
        const int j = j0 + lane / nb;
        const int tb = x.t_lo + j * kWTok + (lane % nb) * btok;
        return (j < ntiles && tb < x.t_hi) ? __ldg(bt + tb / a.P) : 0;
      };
      int cur = load_batch(0), nxt = load_batch(tpb);
      for (int j = 0; j < ntiles; ++j) {
        if (j > 0 && j % tpb == 0) {
          cur = nxt;
          nxt = load_batch(j + tpb);
        }
        const int64_t gg = g + j;
        const int st = (int)(gg % kWStages);
        if (gg >= kWStages && !warp_wait(smem_u32(&bs.stage_empty[st]), ((gg / kWStages) - 1) & 1)) {
          to = true;
          break;
        }
        const int tok0 = x.t_lo + j * kWTok;
        const int nbox = min(nb, (x.t_hi - tok0 + btok - 1) / btok);
        const uint32_t bar = smem_u32(&bs.stage_full[st]);
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nbox * btok * kD));
        __syncwarp();
        int page = __shfl_sync(0xFFFFFFFFu, cur, (j % tpb) * nb + (lane % nb));
        if (lane < nbox) {
          const int tb = tok0 + lane * btok;
          if (page < 0 || (int64_t)page >= a.num_pages) {
            if (!isv) atomicOr(a.status, kErrBadPage);
            page = -1;  // the box lands outside the tensor and reads zeros
          }
          const int row = (page * a.Hkv + x.kvh) * a.P + tb % a.P;
          const uint32_t dst = smem_u32(smem + kWOffStage + st * kWStageBytes) + lane * btok * kD;
          if (isv) tma_load_2d(dst + kWTok * kD, &tmV, 0, row, bar);
          else tma_load_2d(dst, &tmK, 0, row, bar);
        }
      }
      g += ntiles;
      f += ntiles;
    }
    // no copy may still be landing when the CTA retires
    for (int64_t gg = g > kWStages ? g - kWStages : 0; gg < g; ++gg)
      if (!mbar_wait(smem_u32(&bs.stage_full[gg % kWStages]), (gg / kWStages) & 1)) to = true;
  } else if (warp == kWMmaWarp) {
    // ------------------------------------------------- score MMA issuer
    // S(g) = Q . K(g)^T (N = 128) into buffer g % 2, straight from the e4m3 K
    // rows of the stage (kind::f8f6f4: Q in two exact e4m3 parts, four
    // K = 32 steps each), once the stage has landed and the softmax warps have
    // read S(g - 2) from that buffer.  A second commit releases the stage's K;
    // after a unit's last tile a third releases Q.
    if (lane == 0) {
      const uint64_t qdesc = tc::desc_sw128(smem_u32(smem + kWOffQ), 16, 1024);
      int64_t g = 0;
      int k = 0;
      for (int64_t f = f0; f < f1 && !to; ++k) {
        const int ntiles = seg_at(a, f, f1).x.ntiles;
        f += ntiles;
        if (!mbar_wait(smem_u32(&bs.qready), k & 1)) {
          to = true;
          break;
        }
        for (int j = 0; j < ntiles && !to; ++j) {
          const int64_t gg = g + j;
          const int kb = (int)(gg % kWBufs), st = (int)(gg % kWStages);
          if (!mbar_wait(smem_u32(&bs.stage_full[st]), (gg / kWStages) & 1)) to = true;
          if (gg >= kWBufs && !to && !mbar_wait(smem_u32(&bs.sread[kb]), ((gg - kWBufs) / kWBufs) & 1)) to = true;
          if (to) break;
          tc::fence_after_sync();
          const uint64_t kdesc = tc::desc_sw128(smem_u32(smem + kWOffStage + st * kWStageBytes), 16, 1024);
#pragma unroll
          for (int p = 0; p < 2; ++p)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_ss_e4m3(tmem + kWTmemS + kWTok * kb, qdesc + (uint64_t)((p * kWQPart + 32 * kk) >> 4),
                              kdesc + (uint64_t)((32 * kk) >> 4), kIdescQKW, (p > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(smem_u32(&bs.sfull[kb]));
          tc::mma_commit(smem_u32(&bs.stage_empty[st]));
        }
        tc::mma_commit(smem_u32(&bs.qfree));  // Q is free once these products complete
        g += ntiles;
      }
    }
    __syncwarp();
  } else if (warp == kWPvWarp) {
    // ---------------------------------------------------- P.V MMA issuer
    // O += P(g) . V(g) once P and the widened V of tile g are written; a
    // unit's first product overwrites O once the previous unit's epilogue has
    // read it.
    if (lane == 0) {
      const uint32_t v0 = smem_u32(smem + kWOffV);
      int64_t g = 0;
      int k = 0;  // every segment has tiles
      for (int64_t f = f0; f < f1 && !to; ++k) {
        const int ntiles = seg_at(a, f, f1).x.ntiles;
        f += ntiles;
        if (k > 0 && !mbar_wait(smem_u32(&bs.oread), (k - 1) & 1)) {
          to = true;
          break;
        }
        for (int j = 0; j < ntiles && !to; ++j) {
          const int64_t gg = g + j;
          const int kb = (int)(gg % kWBufs);
          if (!mbar_wait(smem_u32(&bs.pfull[kb]), (gg / kWBufs) & 1) ||
              !mbar_wait(smem_u32(&bs.vfull[kb]), (gg / kWBufs) & 1)) {
            to = true;
            break;
          }
          tc::fence_after_sync();
          const uint64_t vdesc = tc::desc_sw128(v0 + kb * kWVBytes, kWAtom, 1024);
#pragma unroll
          for (int kk = 0; kk < kWTok / 16; ++kk)
            tc::mma_ts(tmem + kWTmemO, tmem + kWTmemP + (kWTok / 2) * kb + 8 * kk,
                       vdesc + (uint64_t)((2048 * kk) >> 4), kIdescPVW, (j > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(smem_u32(&bs.pvdone[kb]));
        }
        g += ntiles;
      }
      // every product complete before tensor memory is freed
      if (g > 0 && !mbar_wait(smem_u32(&bs.pvdone[(g - 1) % kWBufs]), ((g - 1) / kWBufs) & 1)) to = true;
    }
    __syncwarp();
  } else if (warp < kWSoftWarp0) {
    // ------------------------------------------------------------ converters
    // V(g): read once the stage has landed, which releases the stage's V at
    // once; written once P.V(g - 2) has completed (its buffer).
    const int ct = threadIdx.x - kWConvWarp0 * 32;
    int64_t g = 0;
    for (int64_t f = f0; f < f1 && !to;) {
      const Seg sg = seg_at(a, f, f1);
      const Unit& x = sg.x;
      const int ntiles = x.ntiles;
      f += ntiles;
      for (int j = 0; j < ntiles; ++j) {
        const int64_t gg = g + j;
        const int st = (int)(gg % kWStages), kb = (int)(gg % kWBufs);
        if (!warp_wait(smem_u32(&bs.stage_full[st]), (gg / kWStages) & 1)) {
          to = true;
          break;
        }
        const int valid = min(kWTok, x.t_hi - (x.t_lo + j * kWTok));
        uint4 v[kWChunks];
        load_v(smem + kWOffStage + st * kWStageBytes + kWTok * kD, ct, valid, v);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.stage_empty[st]));  // release: the reads are done
        if (gg >= kWBufs && !warp_wait(smem_u32(&bs.pvdone[kb]), ((gg - kWBufs) / kWBufs) & 1)) {
          to = true;
          break;
        }
        store_v(v, smem + kWOffV + kb * kWVBytes, ct);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.vfull[kb]));
      }
      g += ntiles;
    }
  } else {
    // -------------------------------------------------- softmax + epilogue
    const int quad = warp & 3;
    const uint32_t trow = tmem + ((uint32_t)(32 * quad) << 16);
    float* const qinv = reinterpret_cast<float*>(smem + kWOffQs);
    // the 16-lane shape: thread t holds row 16 quad + Lm, Lm = (t >> 2) + 8 (t & 1),
    // and the columns of parity par = (t >> 1) & 1 (register k of a 64-column
    // read is column 2 k + par)
    const int Lm = (lane >> 2) + 8 * (lane & 1), par = (lane >> 1) & 1;
    const int rm = 16 * quad + Lm;
    // O row 16 quad + t (t < 16) sits in lane t of the quadrant; its statistics
    // are held by thread 4 (t % 8) + t / 8
    const int src = 4 * (lane & 7) + ((lane >> 3) & 1);
    int64_t g = 0;
    int k = 0;
    for (int64_t f = f0; f < f1 && !to; ++k) {
      const Seg sg = seg_at(a, f, f1);
      const Unit& x = sg.x;
      const int ntiles = x.ntiles;
      f += ntiles;
      // Q: threads t and t + 16 split row 16 quad + t (t < 16), each its half
      // (64 elements), into two e4m3 parts (x = q s with s a power of two
      // taking max |q| of the row into (224, 448]; part 1 = e4m3(x), part 2 =
      // e4m3(x - part 1) = x - part 1), written as the A operands of the score
      // products once the previous unit's products are done; thread t records
      // 1 / s
      if (k > 0 && !warp_wait(smem_u32(&bs.qfree), (k - 1) & 1)) {
        to = true;
        break;
      }
      {
        const int rq = 16 * quad + (lane & 15), hh = lane >> 4;
        const bool okq = rq < x.rows;
        const int64_t hq = ((int64_t)a.q_start[x.b] + x.i0 + rq / a.G) * a.Hq + (int64_t)x.kvh * a.G + rq % a.G;
        const uint4* qp = reinterpret_cast<const uint4*>(a.q + hq * kD) + 8 * hh;
        uint4 qw[8];  // loaded together: one memory latency per unit
#pragma unroll
        for (int uu = 0; uu < 8; ++uu) qw[uu] = okq ? __ldg(qp + uu) : make_uint4(0, 0, 0, 0);
        float amax = 0.f;
#pragma unroll
        for (int uu = 0; uu < 8; ++uu) {
          const uint32_t ww[4] = {qw[uu].x, qw[uu].y, qw[uu].z, qw[uu].w};
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(ww[kk])), fabsf(bf16_hi(ww[kk]))));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 16));  // the row's other half
        // s = 2^floor(log2(448 / amax)) within [2^-126, 2^126] (1 for a zero row)
        const float s = pow2_scale(448.f, amax);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {  // chunk c = 4 hh + cc: 16 elements
          const int c = 4 * hh + cc;
          uint32_t p1[4] = {0u, 0u, 0u, 0u}, p2[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 w = qw[2 * cc + h];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {  // elements 8 h + 2 kk and 8 h + 2 kk + 1 of the chunk
              const float x0 = bf16_lo(ww[kk]) * s, x1 = bf16_hi(ww[kk]) * s;
              const uint16_t c1 = f32x2_to_e4m3x2(x0, x1);
              float d0, d1;
              e4m3x2_to_f32x2(c1, d0, d1);
              const uint16_t c2 = f32x2_to_e4m3x2(x0 - d0, x1 - d1);  // the difference is exact
              const int word = 2 * h + (kk >> 1), sh = 16 * (kk & 1);
              p1[word] |= (uint32_t)c1 << sh;
              p2[word] |= (uint32_t)c2 << sh;
            }
          }
          const uint32_t off = rq * 128 + 16 * (c ^ (rq & 7));  // 128-byte swizzle
          *reinterpret_cast<uint4*>(smem + kWOffQ + off) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
          *reinterpret_cast<uint4*>(smem + kWOffQ + kWQPart + off) = make_uint4(p2[0], p2[1], p2[2], p2[3]);
        }
        if (lane < 16) qinv[rq] = okq ? 1.f / s : 0.f;  // exact: s is a power of two
        fence_proxy_async_smem();  // generic writes -> visible to the tensor core
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.qready));
      }
      const bool okm = rm < x.rows;
      const int im = x.i0 + rm / a.G;
      const int limm = okm ? min(x.L - x.n + im + 1, x.t_end_chunk) : x.t_lo;
      const float sc = a.score_scale * qinv[rm];  // the scores carry the row's Q scale s
      float mref = -INFINITY, rthr = -INFINITY, lpart = 0.f;  // lpart: this thread's share of the row sum
      for (int j = 0; j < ntiles; ++j) {
        const int64_t gg = g + j;
        const int kb = (int)(gg % kWBufs);
        if (!warp_wait(smem_u32(&bs.sfull[kb]), (gg / kWBufs) & 1)) {
          to = true;
          break;
        }
        tc::fence_after_sync();
        // all 128 scores of the row half in registers: sv[32 h + kk] is column
        // 64 h + 2 kk + par; the buffer is then free for S(g + 2)
        uint32_t sv[64];
        {
          uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
          uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
          tc::tmem_ld16x64b_x32(trow + kWTmemS + kWTok * kb, s0);
          tc::tmem_ld16x64b_x32(trow + kWTmemS + kWTok * kb + 64, s1);
          tc::tmem_ld_wait();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.sread[kb]));
        // columns c < nv are attended (none for a padding row); every branch on
        // `full` is warp-uniform and the masks are selects, so no lane diverges
        const int nv = okm ? limm - (x.t_lo + j * kWTok) : 0;
        const bool full = __all_sync(0xFFFFFFFFu, nv >= kWTok);
        float mx;
        {
          float m8[8];
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) m8[kk] = -INFINITY;
          if (full) {
#pragma unroll
            for (int kk = 0; kk < 64; ++kk) m8[kk & 7] = fmaxf(m8[kk & 7], __uint_as_float(sv[kk]));
          } else {
#pragma unroll
            for (int kk = 0; kk < 64; ++kk)
              m8[kk & 7] = fmaxf(m8[kk & 7],
                                 64 * (kk >> 5) + 2 * (kk & 31) + par < nv ? __uint_as_float(sv[kk]) : -INFINITY);
          }
          mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));  // the row's other half
        const bool grow = mx > rthr;
        float al = 1.f;
        bool rescale = false;
        if (__any_sync(0xFFFFFFFFu, grow)) {
          const float mn = grow ? fmaxf(mref, mx * sc) : mref;
          al = grow ? fast_exp2(mref - mn) : 1.f;  // 0 while mref is -inf
          rescale = j > 0 && __any_sync(0xFFFFFFFFu, grow && mref != -INFINITY);
          lpart *= al;
          mref = mn;
          rthr = (mn + kRescaleLog2) / sc;
        }
        // P: register pair (2 r, 2 r + 1) of a half holds tokens (4 r + par, 4 r + par + 2),
        // which the contraction order places in P column 2 r + par of that half
        uint32_t pv[32];
        float ls[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) ls[kk] = 0.f;
        if (full) {
#pragma unroll
          for (int r2 = 0; r2 < 32; ++r2) {
            const float p0 = fast_exp2(fmaf(__uint_as_float(sv[2 * r2]), sc, -mref));
            const float p1 = fast_exp2(fmaf(__uint_as_float(sv[2 * r2 + 1]), sc, -mref));
            ls[r2 & 3] += p0;
            ls[4 + (r2 & 3)] += p1;
            pv[r2] = pack_f16x2(p0, p1);
          }
        } else {
          // a masked column's exponential may overflow; the select drops it
#pragma unroll
          for (int r2 = 0; r2 < 32; ++r2) {
            const int c0 = 64 * (r2 >> 4) + 4 * (r2 & 15) + par;
            const float e0 = fast_exp2(fmaf(__uint_as_float(sv[2 * r2]), sc, -mref));
            const float e1 = fast_exp2(fmaf(__uint_as_float(sv[2 * r2 + 1]), sc, -mref));
            const float p0 = c0 < nv ? e0 : 0.f, p1 = c0 + 2 < nv ? e1 : 0.f;
            ls[r2 & 3] += p0;
            ls[4 + (r2 & 3)] += p1;
            pv[r2] = pack_f16x2(p0, p1);
          }
        }
        lpart += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        // P buffer g % 2 is free once P.V(g - 2) has completed; O, for a
        // rescale, once P.V(g - 1) has (every earlier product is then applied)
        if (gg >= kWBufs || rescale) {
          const int64_t gw = rescale ? gg - 1 : gg - kWBufs;
          if (!warp_wait(smem_u32(&bs.pvdone[gw % kWBufs]), (gw / kWBufs) & 1)) {
            to = true;
            break;
          }
          tc::fence_after_sync();
        }
        if (rescale) {
          // thread t < 16 rescales O row 16 quad + t
          const float alo = __shfl_sync(0xFFFFFFFFu, al, src);
#pragma unroll
          for (int blk = 0; blk < 4; ++blk) {
            uint32_t ov[32];
            tc::tmem_ld32(trow + kWTmemO + 32 * blk, ov);
            tc::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alo);
            tc::tmem_st32(trow + kWTmemO + 32 * blk, ov);
          }
        }
        const uint32_t pbuf = trow + kWTmemP + (kWTok / 2) * kb;
        tc::tmem_st16x64b_x16(pbuf, *reinterpret_cast<const uint32_t(*)[16]>(&pv[0]));
        tc::tmem_st16x64b_x16(pbuf + 32, *reinterpret_cast<const uint32_t(*)[16]>(&pv[16]));
        tc::tmem_st_wait();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.pfull[kb]));
      }
      if (to) break;
      // ---- epilogue: thread t < 16 writes row 16 quad + t from lane t of O
      const float lrow = lpart + __shfl_xor_sync(0xFFFFFFFFu, lpart, 2);
      const float le = __shfl_sync(0xFFFFFFFFu, lrow, src), me = __shfl_sync(0xFFFFFFFFu, mref, src);
      if (ntiles > 0 && !warp_wait(smem_u32(&bs.pvdone[(g + ntiles - 1) % kWBufs]),
                                   ((g + ntiles - 1) / kWBufs) & 1)) {
        to = true;
        break;
      }
      tc::fence_after_sync();
      const int re = 16 * quad + (lane & 15);
      const bool oke = lane < 16 && re < x.rows;
      const int ie = x.i0 + re / a.G, ge = re % a.G;
      const int64_t hre = ((int64_t)a.q_start[x.b] + ie) * a.Hq + (int64_t)x.kvh * a.G + ge;
      const bool direct = sg.whole;
      float* part = direct ? nullptr : a.partials + ((sg.slot * kWRows) + re) * kPartStride;
      const float inv = le > 0.f ? a.out_scale / le : 0.f;
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        uint32_t ov[32];
        if (ntiles > 0) {
          tc::tmem_ld32(trow + kWTmemO + 32 * blk, ov);
          tc::tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = 0u;
        }
        if (!oke) continue;
        if (direct) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = pack_bf16x2(__uint_as_float(ov[2 * c]) * inv, __uint_as_float(ov[2 * c + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + hre * kD + 32 * blk);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            dst[kk] = make_uint4(pk[4 * kk], pk[4 * kk + 1], pk[4 * kk + 2], pk[4 * kk + 3]);
        } else {
          float4* dst = reinterpret_cast<float4*>(part + 4 + 32 * blk);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            dst[kk] = make_float4(__uint_as_float(ov[4 * kk]), __uint_as_float(ov[4 * kk + 1]),
                                  __uint_as_float(ov[4 * kk + 2]), __uint_as_float(ov[4 * kk + 3]));
        }
      }
      if (oke) {
        if (direct) {
          if (a.lse) a.lse[hre] = le > 0.f ? (me + __log2f(le)) * kLn2 : -INFINITY;
        } else {
          part[0] = me;
          part[1] = le;
        }
      }
      // O has been read: the next segment's first P.V may overwrite it
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.oread));
      g += ntiles;
    }
  }

  if (to) atomicOr(a.status, kErrWaitTimeout);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kWMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// One warp per row of a (request, KV head, row block): folds the chunks'
// partial states, M = max m_c, out = sum 2^(m_c - M) o_c / sum 2^(m_c - M) l_c.
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(kMergeWarps * 32) prefill_merge_kernel(const PrefillArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t blk = blockIdx.x / (kRows / kMergeWarps);
  const int r = (int)(blockIdx.x % (kRows / kMergeWarps)) * kMergeWarps + warp;
  const int qb = (int)(blk % a.QB);
  const int64_t bk = blk / a.QB;  // b * Hkv + kvh
  const int64_t u0 = bk * a.C * a.QB + qb;  // unit of chunk 0
  const Unit x = unit_of(a, u0, false);
  if (!x.active || r >= x.rows) return;
  const int nchunks = (x.L + a.split - 1) / a.split;
  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = 0; c < nchunks; ++c) {
    const float* p = a.partials + ((u0 + (int64_t)c * a.QB) * kRows + r) * kPartStride;
    const float mk = p[0], lk = p[1];
    if (lk == 0.f) continue;  // a chunk this row does not reach
    const float4 ok = reinterpret_cast<const float4*>(p + 4)[lane];
    const float Mn = fmaxf(M, mk);
    const float al = fast_exp2(M - Mn), wt = fast_exp2(mk - Mn);
    den = den * al + wt * lk;
    acc.x = acc.x * al + wt * ok.x;
    acc.y = acc.y * al + wt * ok.y;
    acc.z = acc.z * al + wt * ok.z;
    acc.w = acc.w * al + wt * ok.w;
    M = Mn;
  }
  const int i = x.i0 + r / a.G, g = r % a.G;
  const int64_t head_row = ((int64_t)a.q_start[x.b] + i) * a.Hq + (int64_t)x.kvh * a.G + g;
  const float inv = den > 0.f ? a.out_scale / den : 0.f;
  reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + head_row * kD)[lane] =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (a.lse && lane == 0) a.lse[head_row] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
}

// One warp per row of a (request, KV head) on the flattened path: folds the
// partial states of the CTAs whose tile ranges cut the pair's range (slot
// CTA + pair), in CTA order, skipping CTAs whose range is empty; a pair
// inside one CTA's range was written by it.
__global__ void __launch_bounds__(kMergeWarps * 32) prefillw_merge_kernel(const PrefillArgs a) {
  grid_dependency_wait();  // every partial state of the tile kernel is visible
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t u = blockIdx.x / (kWRows / kMergeWarps);
  const int r = (int)(blockIdx.x % (kWRows / kMergeWarps)) * kMergeWarps + warp;
  const int b = (int)(u / a.Hkv), kvh = (int)(u % a.Hkv);
  const int64_t s0 = a.tile_start[b];
  const int64_t per = (a.tile_start[b + 1] - s0) / a.Hkv;
  if (per == 0) return;
  int L, n;
  clamped_ln(a, b, L, n, false);
  if (r >= n * a.G) return;
  const int64_t W = a.tile_start[a.B], N = a.ncta;
  const int64_t T0 = s0 + kvh * per, T1 = T0 + per;
  const int64_t i0 = ((T0 + 1) * N - 1) / W, i1 = (T1 * N - 1) / W;  // owners of tiles T0 and T1 - 1
  if (i0 == i1) return;
  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t i = i0; i <= i1; ++i) {
    if (i * W / N == (i + 1) * W / N) continue;  // an empty range (fewer tiles than CTAs) wrote nothing
    const float* p = a.partials + ((i + u) * kWRows + r) * kPartStride;
    const float mk = p[0], lk = p[1];
    if (lk == 0.f) continue;  // a run this row does not reach
    const float4 ok = reinterpret_cast<const float4*>(p + 4)[lane];
    const float Mn = fmaxf(M, mk);
    const float al = fast_exp2(M - Mn), wt = fast_exp2(mk - Mn);
    den = den * al + wt * lk;
    acc.x = acc.x * al + wt * ok.x;
    acc.y = acc.y * al + wt * ok.y;
    acc.z = acc.z * al + wt * ok.z;
    acc.w = acc.w * al + wt * ok.w;
    M = Mn;
  }
  const int64_t head_row = ((int64_t)a.q_start[b] + r / a.G) * a.Hq + (int64_t)kvh * a.G + r % a.G;
  const float inv = den > 0.f ? a.out_scale / den : 0.f;
  reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(a.out) + head_row * kD)[lane] =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (a.lse && lane == 0) a.lse[head_row] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
}

// ------------------------------------- one 128-row block per CTA, Q in TMEM
// For row blocks of more than 64 rows (chunked prefill), prefillm_kernel
// takes one block of 128 rows per CTA over 128-token tiles, with Q's two
// exact e4m3 parts in tensor memory as the A operand of the score products
// (kind::f8f6f4, M = 128, N = 128), so those products read only the K rows
// from shared memory (an earlier kernel taking two blocks per CTA, with Q in
// shared memory because the two blocks' accumulators filled tensor memory,
// was bound by that operand traffic).  Eight softmax
// warps, two per lane quadrant, each take 64 of a row's 128 scores: the two
// halves of a row swap their maxima (and, once per unit, Q's largest
// magnitude and at the end the row sums) through shared memory, handing over
// with an mbarrier per quadrant and bounded waits, so the reference and the
// rescale are the same in both.  P (f16) has 64 tensor-memory columns of its
// own; V rows are widened in token order (a thread packs the columns of its
// row two by two).
//   tensor memory: S 2 x 128, O 128, Q 2 x 32 (part p at 384 + 32 p), P 64.
//   shared memory: three 32 KB e4m3 stages, three 32 KB widened V tiles (a
//   stage is released once its V is read, so three cover the copy latency;
//   the third V tile lets the widening of tile j + 2 run while P.V(j) waits
//   for its P).
//   warps: 0 K producer, 1 score MMAs, 2-5 widening, 6-13 softmax (warp w:
//   lane quadrant w % 4, half (w - 6) / 4), 14 P.V MMAs, 15 V producer (one
//   warp issuing every copy of a tile measured slower, most of all with
//   16-token pages: 16 copies per tile; so did one thread issuing both kinds
//   of MMA, by 25%: the two issuers' MMAs overlap their latencies).
// Units in order of decreasing row block, so the longest (causal) ones start first.
// Score and P buffers in tensor memory.  One score buffer and two P buffers
// (so that P(j + 1) need not wait for P.V(j)) fit as well and give the same
// output, but measured 0.5-1% slower: S(j + 1) then waits for the softmax
// to read S(j), a loop of the same length.
constexpr int kMSBufs = 2, kMPBufs = 1;
constexpr int kMTmemO = kMSBufs * kWTok, kMTmemQ = kMTmemO + kD, kMTmemP = kMTmemQ + 64;
static_assert(kMTmemP + kMPBufs * kWTok / 2 <= kTmemCols, "tensor memory columns");
constexpr int kMStages = 3, kMVBufs = 3;
constexpr int kMOffV = 0;
constexpr int kMOffStage = kMOffV + kMVBufs * kWVBytes;
constexpr int kMOffX = kMOffStage + kMStages * kWStageBytes;  // float [2 parity][2 halves][128 rows]
constexpr int kMOffBars = kMOffX + 2 * 2 * kRows * 4;
constexpr int kMSmemBytes = kMOffBars + 512 + 1024;
static_assert(kMSmemBytes <= 232448, "shared memory over the per-CTA limit");
constexpr uint32_t kIdescQKM = tc::idesc_f16(kRows, kWTok, false);  // with kind::f8f6f4: e4m3 x e4m3
constexpr uint32_t kIdescPVM = tc::idesc_f16(kRows, kD, true);
constexpr int kMProdWarp = 0, kMMmaWarp = 1, kMConvWarp0 = 2, kMSoftWarp0 = 6, kMPvWarp = 14, kMProdWarpV = 15;
constexpr int kMThreads = 16 * 32;

struct BarsM {
  uint64_t stage_full[kMStages], stage_empty[kMStages];
  uint64_t vfull[kMVBufs], vfree[kMVBufs];  // widened V written / read by its P.V
  uint64_t sfull[kMSBufs], sread[kMSBufs], pfull[kMPBufs], pvdone[kMPBufs];
  uint64_t qready;
  uint64_t xch[4];  // the two softmax warps of a lane quadrant hand over shared values
  uint32_t tmem_base;
};
static_assert(sizeof(BarsM) <= 512, "barrier block");

// As store_v, rows in token order.
__device__ __forceinline__ void store_v_tokens(const uint4 (&v)[kWChunks], uint8_t* dst, int ct) {
#pragma unroll
  for (int m = 0; m < kWChunks; ++m) {
    const int i = ct + 32 * kWConvWarps * m;
    const int row = i >> 3, c = i & 7;
    uint4 o0, o1;
    e4m3x4_to_f16x2x2(v[m].x, o0.x, o0.y);
    e4m3x4_to_f16x2x2(v[m].y, o0.z, o0.w);
    e4m3x4_to_f16x2x2(v[m].z, o1.x, o1.y);
    e4m3x4_to_f16x2x2(v[m].w, o1.z, o1.w);
    const uint32_t d = atom_off(row, 2 * c, kWAtom);
    *reinterpret_cast<uint4*>(dst + d) = o0;
    *reinterpret_cast<uint4*>(dst + (d ^ 16)) = o1;
  }
}

__global__ void __launch_bounds__(kMThreads, 1)
    prefillm_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* const smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  BarsM& bs = *reinterpret_cast<BarsM*>(smem + kMOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // CTA -> unit: row blocks from the last (longest under the causal mask) down
  const int64_t per_qb = (int64_t)a.B * a.Hkv * a.C;
  const int qb = a.QB - 1 - (int)(blockIdx.x / per_qb);
  const int64_t u = (blockIdx.x % per_qb) * a.QB + qb;
  const Unit x = unit_of(a, u, threadIdx.x == 0 && qb == 0 && (u / a.QB) % ((int64_t)a.C * a.Hkv) == 0);
  if (!x.active) return;  // uniform over the CTA
  const int ntiles = x.ntiles == 0 ? 0 : (x.t_hi - x.t_lo + kWTok - 1) / kWTok;
  const bool direct = a.C == 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMStages; ++s) {
      mbar_init(smem_u32(&bs.stage_full[s]), 2);  // the K and the V producer
      mbar_init(smem_u32(&bs.stage_empty[s]), kWConvWarps + 1);  // V read + the score products done
    }
    for (int k = 0; k < kMVBufs; ++k) {
      mbar_init(smem_u32(&bs.vfull[k]), kWConvWarps);
      mbar_init(smem_u32(&bs.vfree[k]), 1);
    }
    for (int k = 0; k < kMSBufs; ++k) {
      mbar_init(smem_u32(&bs.sfull[k]), 1);
      mbar_init(smem_u32(&bs.sread[k]), 8);
    }
    for (int k = 0; k < kMPBufs; ++k) {
      mbar_init(smem_u32(&bs.pfull[k]), 8);
      mbar_init(smem_u32(&bs.pvdone[k]), 1);
    }
    mbar_init(smem_u32(&bs.qready), 8);
    for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&bs.xch[q]), 2);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (warp == kMMmaWarp) {
    tc::tmem_alloc(smem_u32(&bs.tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bs.tmem_base;
  bool to = false;  // a bounded wait gave up

  if (warp == kMProdWarp || warp == kMProdWarpV) {
    // ------------------------------------------------------------ producers
    // as in prefillw_kernel: nb boxes of box_tok rows per tensor and tile;
    // warp kMProdWarp copies K, warp kMProdWarpV copies V, each arriving on
    // the stage with its own byte count
    const bool isv = warp == kMProdWarpV;
    const int btok = a.box_tok, nb = kWTok / btok, tpb = 32 / nb;
    const int32_t* bt = a.block_tables + (int64_t)x.b * a.max_pages;
    auto load_batch = [&](int j0) {
      const int j = j0 + lane / nb;
      const int tb = x.t_lo + j * kWTok + (lane % nb) * btok;
      return (j < ntiles && tb < x.t_hi) ? __ldg(bt + tb / a.P) : 0;
    };
    int cur = load_batch(0), nxt = load_batch(tpb);
    for (int j = 0; j < ntiles && !to; ++j) {
      if (j > 0 && j % tpb == 0) {
        cur = nxt;
        nxt = load_batch(j + tpb);
      }
      const int st = j % kMStages;
      if (j >= kMStages && !warp_wait(smem_u32(&bs.stage_empty[st]), ((j / kMStages) - 1) & 1)) {
        to = true;
        break;
      }
      const int tok0 = x.t_lo + j * kWTok;
      const int nbox = min(nb, (x.t_hi - tok0 + btok - 1) / btok);
      const uint32_t bar = smem_u32(&bs.stage_full[st]);
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nbox * btok * kD));
      __syncwarp();
      int page = __shfl_sync(0xFFFFFFFFu, cur, (j % tpb) * nb + (lane % nb));
      if (lane < nbox) {
        const int tb = tok0 + lane * btok;
        if (page < 0 || (int64_t)page >= a.num_pages) {
          if (!isv) atomicOr(a.status, kErrBadPage);
          page = -1;  // the box lands outside the tensor and reads zeros
        }
        const int row = (page * a.Hkv + x.kvh) * a.P + tb % a.P;
        const uint32_t dst = smem_u32(smem + kMOffStage + st * kWStageBytes) + lane * btok * kD;
        if (isv) tma_load_2d(dst + kWTok * kD, &tmV, 0, row, bar);
        else tma_load_2d(dst, &tmK, 0, row, bar);
      }
    }
    for (int j = ntiles > kMStages ? ntiles - kMStages : 0; j < ntiles; ++j)
      if (!mbar_wait(smem_u32(&bs.stage_full[j % kMStages]), (j / kMStages) & 1)) to = true;
  } else if (warp == kMMmaWarp) {
    // ------------------------------------------------- score MMA issuer
    // S(j) = Q . K(j)^T (M = N = 128) into buffer j % 2, Q's two e4m3 parts
    // from tensor memory (four K = 32 steps each), once the stage has landed
    // and the softmax warps have read S(j - 2); a second commit releases K.
    if (lane == 0 && ntiles > 0) {
      if (!mbar_wait(smem_u32(&bs.qready), 0)) to = true;
      for (int j = 0; j < ntiles && !to; ++j) {
        const int kb = j % kMSBufs, st = j % kMStages;
        if (!mbar_wait(smem_u32(&bs.stage_full[st]), (j / kMStages) & 1)) to = true;
        if (j >= kMSBufs && !to && !mbar_wait(smem_u32(&bs.sread[kb]), ((j - kMSBufs) / kMSBufs) & 1)) to = true;
        if (to) break;
        tc::fence_after_sync();
        const uint64_t kdesc = tc::desc_sw128(smem_u32(smem + kMOffStage + st * kWStageBytes), 16, 1024);
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_ts_e4m3(tmem + kWTok * kb, tmem + kMTmemQ + 32 * p + 8 * kk, kdesc + (uint64_t)((32 * kk) >> 4),
                            kIdescQKM, (p > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(smem_u32(&bs.sfull[kb]));
        tc::mma_commit(smem_u32(&bs.stage_empty[st]));
      }
    }
    __syncwarp();
  } else if (warp == kMPvWarp) {
    // ---------------------------------------------------- P.V MMA issuer
    if (lane == 0 && ntiles > 0) {
      const uint32_t v0 = smem_u32(smem + kMOffV);
      int pn = 0;
      for (; pn < ntiles && !to; ++pn) {
        const int kb = pn % kMPBufs, vb = pn % kMVBufs;
        if (!mbar_wait(smem_u32(&bs.pfull[kb]), (pn / kMPBufs) & 1) ||
            !mbar_wait(smem_u32(&bs.vfull[vb]), (pn / kMVBufs) & 1)) {
          to = true;
          break;
        }
        tc::fence_after_sync();
        const uint64_t vdesc = tc::desc_sw128(v0 + vb * kWVBytes, kWAtom, 1024);
#pragma unroll
        for (int kk = 0; kk < kWTok / 16; ++kk)
          tc::mma_ts(tmem + kMTmemO, tmem + kMTmemP + 64 * kb + 8 * kk, vdesc + (uint64_t)((2048 * kk) >> 4), kIdescPVM,
                     (pn > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(smem_u32(&bs.pvdone[kb]));
        tc::mma_commit(smem_u32(&bs.vfree[vb]));
      }
      if (pn > 0 && !mbar_wait(smem_u32(&bs.pvdone[(pn - 1) % kMPBufs]), ((pn - 1) / kMPBufs) & 1)) to = true;
    }
    __syncwarp();
  } else if (warp < kMSoftWarp0) {
    // ------------------------------------------------------------ converters
    const int ct = threadIdx.x - kMConvWarp0 * 32;
    for (int j = 0; j < ntiles && !to; ++j) {
      const int st = j % kMStages, vb = j % kMVBufs;
      if (!warp_wait(smem_u32(&bs.stage_full[st]), (j / kMStages) & 1)) {
        to = true;
        break;
      }
      const int valid = min(kWTok, x.t_hi - (x.t_lo + j * kWTok));
      uint4 v[kWChunks];
      load_v(smem + kMOffStage + st * kWStageBytes + kWTok * kD, ct, valid, v);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.stage_empty[st]));  // release: the reads are done
      if (j >= kMVBufs && !warp_wait(smem_u32(&bs.vfree[vb]), ((j - kMVBufs) / kMVBufs) & 1)) {
        to = true;
        break;
      }
      store_v_tokens(v, smem + kMOffV + vb * kWVBytes, ct);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.vfull[vb]));
    }
  } else {
    // -------------------------------------------------- softmax + epilogue
    const int quad = warp & 3, half = (warp - kMSoftWarp0) >> 2;
    const int r = 32 * quad + lane;  // this thread's row; columns 64 half .. 64 half + 63
    const uint32_t trow = tmem + ((uint32_t)(32 * quad) << 16);
    const bool row_ok = r < x.rows;
    const int i = x.i0 + r / a.G, g = r % a.G;
    const int64_t head_row = ((int64_t)a.q_start[x.b] + i) * a.Hq + (int64_t)x.kvh * a.G + g;
    float* const xv = reinterpret_cast<float*>(smem + kMOffX);  // [parity][half][row]
    const uint32_t xbar = smem_u32(&bs.xch[quad]);
    int ex = 0;  // exchanges so far (the barrier's phase)
    // hand this half's value for row r to the other half and return the other's
    auto swap = [&](float val) -> float {
      xv[((ex & 1) * 2 + half) * kRows + r] = val;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(xbar);
      if (!warp_wait(xbar, ex & 1)) to = true;
      const float other = xv[((ex & 1) * 2 + (half ^ 1)) * kRows + r];
      ++ex;
      return other;
    };
    // Q: this half's 64 elements of row r as two exact e4m3 parts (x = q s, s
    // = 2^floor(log2(448 / max |q|)) over the whole row; part 1 = e4m3(x),
    // part 2 = e4m3(x - part 1)) into tensor memory, K order, four per column
    float qinv;
    {
      const uint4* qp = reinterpret_cast<const uint4*>(a.q + head_row * kD) + 8 * half;
      uint4 qw[8];
#pragma unroll
      for (int uu = 0; uu < 8; ++uu) qw[uu] = row_ok ? __ldg(qp + uu) : make_uint4(0, 0, 0, 0);
      float amax = 0.f;
#pragma unroll
      for (int uu = 0; uu < 8; ++uu) {
        const uint32_t ww[4] = {qw[uu].x, qw[uu].y, qw[uu].z, qw[uu].w};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(ww[kk])), fabsf(bf16_hi(ww[kk]))));
      }
      amax = fmaxf(amax, swap(amax));
      const float s = pow2_scale(448.f, amax);
      qinv = row_ok ? 1.f / s : 0.f;  // exact: s is a power of two
      uint32_t p1[16], p2[16];
#pragma unroll
      for (int uu = 0; uu < 8; ++uu) {
        const uint32_t ww[4] = {qw[uu].x, qw[uu].y, qw[uu].z, qw[uu].w};
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {  // elements 8 uu + 4 h2 .. + 3: one column
          uint32_t c1w = 0u, c2w = 0u;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t w = ww[2 * h2 + e];
            const float x0 = bf16_lo(w) * s, x1 = bf16_hi(w) * s;
            const uint16_t c1 = f32x2_to_e4m3x2(x0, x1);
            float d0, d1;
            e4m3x2_to_f32x2(c1, d0, d1);
            const uint16_t c2 = f32x2_to_e4m3x2(x0 - d0, x1 - d1);  // the difference is exact
            c1w |= (uint32_t)c1 << (16 * e);
            c2w |= (uint32_t)c2 << (16 * e);
          }
          p1[2 * uu + h2] = c1w;
          p2[2 * uu + h2] = c2w;
        }
      }
      tc::tmem_st16(trow + kMTmemQ + 16 * half, p1);
      tc::tmem_st16(trow + kMTmemQ + 32 + 16 * half, p2);
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.qready));
    }
    const int lim = row_ok ? min(x.L - x.n + i + 1, x.t_end_chunk) : x.t_lo;
    const float sc = a.score_scale * qinv;  // the scores carry the row's Q scale
    float mref = -INFINITY, rthr = -INFINITY, lpart = 0.f;
    for (int j = 0; j < ntiles && !to; ++j) {
      const int kb = j % kMSBufs, pb = j % kMPBufs;
      if (!warp_wait(smem_u32(&bs.sfull[kb]), (j / kMSBufs) & 1)) {
        to = true;
        break;
      }
      tc::fence_after_sync();
      const uint32_t sbase = trow + kWTok * kb + 64 * half;
      const int nv = lim - (x.t_lo + j * kWTok + 64 * half);  // this half's columns c < nv are attended
      const bool full = __all_sync(0xFFFFFFFFu, nv >= 64);
      // this half's 64 scores in registers at once; the buffer is then free for S(j + kMSBufs)
      uint32_t sv[64];
      {
        uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
        uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
        tc::tmem_ld32(sbase, s0);
        tc::tmem_ld32(sbase + 32, s1);
        tc::tmem_ld_wait();
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.sread[kb]));
      float mx;
      {
        float m8[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) m8[kk] = -INFINITY;
        if (full) {
#pragma unroll
          for (int c = 0; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], __uint_as_float(sv[c]));
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], c < nv ? __uint_as_float(sv[c]) : -INFINITY);
        }
        mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      }
      mx = fmaxf(mx, swap(mx));  // the row's maximum, the same in both halves
      if (to) break;
      const bool grow = mx > rthr;
      float al = 1.f;
      bool rescale = false;
      if (__any_sync(0xFFFFFFFFu, grow)) {
        const float mn = grow ? fmaxf(mref, mx * sc) : mref;
        al = grow ? fast_exp2(mref - mn) : 1.f;  // 0 while mref is -inf
        rescale = j > 0 && __any_sync(0xFFFFFFFFu, grow && mref != -INFINITY);
        lpart *= al;
        mref = mn;
        rthr = (mn + kRescaleLog2) / sc;
      }
      // P for this half (column pair c -> word c / 2 of 32)
      uint32_t pv[32];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      if (full) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float x1 = fmaf(__uint_as_float(sv[2 * c + 1]), sc, -mref);
          const float p0 = fast_exp2(fmaf(__uint_as_float(sv[2 * c]), sc, -mref));
          const float p1 = fast_exp2(x1);
          ls[c & 3] += p0 + p1;
          pv[c] = pack_f16x2(p0, p1);
        }
      } else {
        // a masked column's exponential may overflow; the select drops it
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float x1 = fmaf(__uint_as_float(sv[2 * c + 1]), sc, -mref);
          const float e0 = fast_exp2(fmaf(__uint_as_float(sv[2 * c]), sc, -mref));
          const float e1 = fast_exp2(x1);
          const float p0 = 2 * c < nv ? e0 : 0.f, p1 = 2 * c + 1 < nv ? e1 : 0.f;
          ls[c & 3] += p0 + p1;
          pv[c] = pack_f16x2(p0, p1);
        }
      }
      lpart += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      // P buffer pb is free once P.V(j - kMPBufs) has completed, O once P.V(j - 1) has
      if (j >= kMPBufs || (rescale && kMPBufs > 1)) {
        const int jw = rescale ? j - 1 : j - kMPBufs;  // the later of the two when both apply
        if (!warp_wait(smem_u32(&bs.pvdone[jw % kMPBufs]), (jw / kMPBufs) & 1)) {
          to = true;
          break;
        }
        tc::fence_after_sync();
      }
      if (rescale) {  // this half's 64 columns of O for the warp's rows
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          uint32_t ov[32];
          tc::tmem_ld32(trow + kMTmemO + 64 * half + 32 * blk, ov);
          tc::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * al);
          tc::tmem_st32(trow + kMTmemO + 64 * half + 32 * blk, ov);
        }
      }
      tc::tmem_st32(trow + kMTmemP + 64 * pb + 32 * half, pv);
      tc::tmem_st_wait();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_local(smem_u32(&bs.pfull[pb]));
    }
    // ---- epilogue: this half's 64 columns of row r
    if (!to) {
      const float l = lpart + swap(lpart);
      if (!to && ntiles > 0 &&
          !warp_wait(smem_u32(&bs.pvdone[(ntiles - 1) % kMPBufs]), ((ntiles - 1) / kMPBufs) & 1))
        to = true;
      tc::fence_after_sync();
      float* part = direct ? nullptr : a.partials + (u * kRows + r) * kPartStride;
      const float inv = l > 0.f ? a.out_scale / l : 0.f;
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        uint32_t ov[32];
        if (ntiles > 0) {
          tc::tmem_ld32(trow + kMTmemO + 64 * half + 32 * blk, ov);
          tc::tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = 0u;
        }
        if (!row_ok || to) continue;
        const int d0 = 64 * half + 32 * blk;  // head_dim columns d0 .. d0 + 31
        if (direct) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = pack_bf16x2(__uint_as_float(ov[2 * c]) * inv, __uint_as_float(ov[2 * c + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + head_row * kD + d0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) dst[kk] = make_uint4(pk[4 * kk], pk[4 * kk + 1], pk[4 * kk + 2], pk[4 * kk + 3]);
        } else {
          float4* dst = reinterpret_cast<float4*>(part + 4 + d0);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            dst[kk] = make_float4(__uint_as_float(ov[4 * kk]), __uint_as_float(ov[4 * kk + 1]),
                                  __uint_as_float(ov[4 * kk + 2]), __uint_as_float(ov[4 * kk + 3]));
        }
      }
      if (row_ok && !to && half == 0) {
        if (direct) {
          if (a.lse) a.lse[head_row] = l > 0.f ? (mref + __log2f(l)) * kLn2 : -INFINITY;
        } else {
          part[0] = mref;
          part[1] = l;
        }
      }
    }
  }

  if (to) atomicOr(a.status, kErrWaitTimeout);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

constexpr size_t kStatusBytes = 256;

int64_t units_of(int B, int Hkv, int QB, int C) { return (int64_t)B * Hkv * QB * C; }

// The flattened path (every block at most 64 rows): the request offsets, then
// one 64-row partial state per (CTA, pair) slot, CTAs + B Hkv slots.
size_t wide_offsets_bytes(int B) { return ((size_t)(B + 1) * sizeof(int64_t) + 255) / 256 * 256; }
size_t wide_workspace_bytes(int B, int Hkv) {
  const int ncta = device_sm_count() > 0 ? device_sm_count() : 1;
  return kStatusBytes + wide_offsets_bytes(B) +
         ((size_t)ncta + (size_t)B * Hkv) * kWRows * kPartStride * sizeof(float);
}

}  // namespace
}  // namespace pfkv

extern "C" {

size_t pfkv_paged_prefill_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                         int max_q_len, int max_context_len, int kv_split_tokens) {
  using namespace pfkv;
  (void)head_dim;
  if (batch < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads || max_q_len <= 0 ||
      max_context_len <= 0 || kv_split_tokens < 0)
    return 0;
  const int G = num_q_heads / num_kv_heads;
  if (G > kRows) return 0;
  const int QB = (int)(((int64_t)max_q_len * G + kRows - 1) / kRows);
  if ((int64_t)max_q_len * G <= kWRows) return wide_workspace_bytes(batch, num_kv_heads);
  const int C = kv_split_tokens > 0 ? (max_context_len + kv_split_tokens - 1) / kv_split_tokens : 1;
  if (C <= 1) return kStatusBytes;
  return kStatusBytes + (size_t)units_of(batch, num_kv_heads, QB, C) * kRows * kPartStride * sizeof(float);
}

int pfkv_paged_prefill_attn(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_pages_per_seq, const int32_t* context_lens,
                            const int32_t* q_start, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                            int page_size, int64_t num_pages, int max_q_len, int max_context_len, float k_scale,
                            float v_scale, float softmax_scale, int kv_split_tokens, void* workspace,
                            size_t workspace_bytes, float* lse_out, pfkv_stream_t stream) {
  using namespace pfkv;
  clear_error();
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || page_size <= 0 || num_pages <= 0 ||
      max_pages_per_seq <= 0 || max_q_len <= 0 || max_context_len <= 0)
    return fail(PFKV_ERR_INVALID_ARG, "paged_prefill: bad sizes");
  if (num_q_heads % num_kv_heads != 0)
    return fail(PFKV_ERR_INVALID_ARG, "paged_prefill: num_q_heads %% num_kv_heads != 0");
  const int G = num_q_heads / num_kv_heads;
  if (kRows % G != 0)
    return fail(PFKV_ERR_UNSUPPORTED, "paged_prefill: group size %d does not divide 128", G);
  if (head_dim != kD) return fail(PFKV_ERR_UNSUPPORTED, "paged_prefill: head_dim %d != 128", head_dim);
  if (page_size % kBoxTok != 0)
    return fail(PFKV_ERR_UNSUPPORTED, "paged_prefill: page_size %d not a multiple of 16", page_size);
  if (kv_split_tokens < 0 || kv_split_tokens % kTokN != 0)
    return fail(PFKV_ERR_INVALID_ARG, "paged_prefill: kv_split_tokens must be a multiple of 64");
  if ((int64_t)num_pages * num_kv_heads * page_size >= (int64_t)1 << 31)
    return fail(PFKV_ERR_UNSUPPORTED, "paged_prefill: cache has 2^31 or more token rows");
  if ((int64_t)max_pages_per_seq * page_size >= (int64_t)1 << 30 || max_context_len >= (1 << 30))
    return fail(PFKV_ERR_UNSUPPORTED, "paged_prefill: context too long");
  if (!(softmax_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale) || !isfinite(softmax_scale))
    return fail(PFKV_ERR_INVALID_ARG, "paged_prefill: scales must be finite");
  if (batch == 0) return PFKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !q_start || !workspace)
    return fail(PFKV_ERR_INVALID_ARG, "paged_prefill: null pointer");
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(workspace, 256) || !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
      !aligned(q_start, 4) || (lse_out && !aligned(lse_out, 4)))
    return fail(PFKV_ERR_INVALID_ARG, "paged_prefill: misaligned pointer");
  const size_t need = pfkv_paged_prefill_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_q_len,
                                                        max_context_len, kv_split_tokens);
  if (need == 0 || workspace_bytes < need)
    return fail(PFKV_ERR_WORKSPACE, "paged_prefill: workspace of %zu bytes is too small (%zu needed)",
                workspace_bytes, need);

  PrefillArgs a;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.q_start = q_start;
  a.lse = lse_out;
  a.status = reinterpret_cast<int32_t*>(ws);
  a.partials = reinterpret_cast<float*>(ws + kStatusBytes);
  a.B = batch;
  a.Hq = num_q_heads;
  a.Hkv = num_kv_heads;
  a.G = G;
  a.P = page_size;
  a.max_pages = max_pages_per_seq;
  a.QB = (int)(((int64_t)max_q_len * G + kRows - 1) / kRows);
  a.C = kv_split_tokens > 0 ? (max_context_len + kv_split_tokens - 1) / kv_split_tokens : 1;
  a.split = kv_split_tokens > 0 ? kv_split_tokens : (1 << 30);
  a.max_q_len = max_q_len;
  a.max_ctx = max_context_len;
  a.num_pages = num_pages;
  a.score_scale = k_scale * softmax_scale * kLog2e;
  a.out_scale = v_scale;
  a.box_tok = kBoxTok;
  const int64_t units = units_of(batch, num_kv_heads, a.QB, a.C);
  if (units > 0x7FFFFFFF) return fail(PFKV_ERR_UNSUPPORTED, "paged_prefill: too many work units");

  const cuuint64_t rows = (cuuint64_t)num_pages * num_kv_heads * page_size;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, (cuuint32_t)kBoxTok};
  CUtensorMap tmK, tmV;
  int rc = encode_tensor_map(&tmK, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(k_cache), dims, strides,
                             box, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == PFKV_OK)
    rc = encode_tensor_map(&tmV, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(v_cache), dims, strides,
                           box, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != PFKV_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(a.status, 0, sizeof(int32_t), s) != cudaSuccess) return check_cuda("paged_prefill status");
  // both kernels take 128-token tiles as boxes as tall as the page allows
  // (up to 64 rows): fewer copies per tile
  a.box_tok = page_size % 64 == 0 ? 64 : (page_size % 32 == 0 ? 32 : kBoxTok);
  if (a.box_tok != kBoxTok) {
    const cuuint32_t boxw[2] = {128, (cuuint32_t)a.box_tok};
    rc = encode_tensor_map(&tmK, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(k_cache), dims, strides,
                           boxw, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc == PFKV_OK)
      rc = encode_tensor_map(&tmV, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(v_cache), dims, strides,
                             boxw, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != PFKV_OK) return rc;
  }
  if ((int64_t)max_q_len * G <= 64) {
    // every block has at most 64 rows: 128-token tiles, half-height products
    static std::atomic<uint64_t> smemw_set{0};
    rc = set_max_dynamic_smem(reinterpret_cast<const void*>(prefillw_kernel), kWSmemBytes, smemw_set,
                              "paged_prefill set smem attribute");
    if (rc != PFKV_OK) return rc;
    // the KV range of all (request, KV head) pairs split evenly over one CTA
    // per SM (kv_split_tokens is not needed here); plan, tile kernel and merge,
    // the last two as programmatic dependents of the kernel before them
    a.ncta = device_sm_count() > 0 ? device_sm_count() : 1;
    a.tile_start = reinterpret_cast<int64_t*>(ws + kStatusBytes);
    a.partials = reinterpret_cast<float*>(ws + kStatusBytes + wide_offsets_bytes(batch));
    prefillw_plan_kernel<<<1, 1024, 0, s>>>(a);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)a.ncta);
    cfg.blockDim = dim3(kWThreads);
    cfg.dynamicSmemBytes = kWSmemBytes;
    if (cudaLaunchKernelEx(&cfg, prefillw_kernel, tmK, tmV, a) != cudaSuccess) return check_cuda("paged_prefill launch");
    cfg.gridDim = dim3((unsigned)((int64_t)batch * num_kv_heads * (kWRows / kMergeWarps)));
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(&cfg, prefillw_merge_kernel, a) != cudaSuccess) return check_cuda("paged_prefill merge");
    return check_cuda("paged_prefill launch");
  }
  // blocks of up to 128 rows: one per CTA, Q in tensor memory, longest first
  static std::atomic<uint64_t> smemm_set{0};
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(prefillm_kernel), kMSmemBytes, smemm_set,
                            "paged_prefill set smem attribute");
  if (rc != PFKV_OK) return rc;
  prefillm_kernel<<<(unsigned)units, kMThreads, kMSmemBytes, s>>>(tmK, tmV, a);
  if (a.C > 1) {
    const int64_t mblocks = (int64_t)batch * num_kv_heads * a.QB * (kRows / kMergeWarps);
    prefill_merge_kernel<<<(unsigned)mblocks, kMergeWarps * 32, 0, s>>>(a);
  }
  return check_cuda("paged_prefill launch");
}

}  // extern "C"
