// validate.cu -- opt-in batched index check run before decode.
//
// Workers AI post (より小さく、高速で、安全に), §3 "共用 KV キャッシュの保護":
// before decode reads the cache, verify the request-to-page mapping, and do it
// as its own batched check rather than inside the attention kernel so that the
// attention path pays nothing for it.  This kernel checks the index data the
// attention kernels trust: context lengths against the block table, the block
// table entries a request uses against the page pool, top-k indices against the
// context, and slot-mapping entries against the cache.
#include "pfkv_internal.h"
#include "pfkv_ptx.cuh"

namespace pfkv {
namespace {

struct ValidateArgs {
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* topk;
  const int64_t* slots;
  int32_t* err;
  int B, max_pages, P, topk_n, num_slots;
  int64_t num_pages;
};

__global__ void __launch_bounds__(256) validate_kernel(const ValidateArgs a) {
  // blockIdx.y = request b (block-table row and top-k row); the x dimension
  // strides over that row.  Row B (the extra y index) checks the slot mapping.
  const int b = blockIdx.y;
  int bits = 0;
  if (b < a.B) {
    int L = a.context_lens[b];
    if (L < 0 || L > a.max_pages * a.P) {
      bits |= kErrBadContext;
      L = L < 0 ? 0 : a.max_pages * a.P;
    }
    const int used = (L + a.P - 1) / a.P;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < used; i += gridDim.x * blockDim.x) {
      const int page = a.block_tables[(int64_t)b * a.max_pages + i];
      if (page < 0 || page >= a.num_pages) bits |= kErrBadPage;
    }
    if (a.topk) {
      for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.topk_n; i += gridDim.x * blockDim.x) {
        const int t = a.topk[(int64_t)b * a.topk_n + i];
        if (t >= L) bits |= kErrBadTopk;
      }
    }
  } else if (a.slots) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.num_slots; i += gridDim.x * blockDim.x) {
      const int64_t s = a.slots[i];
      if (s >= a.num_pages * (int64_t)a.P) bits |= kErrBadSlot;
    }
  }
  // one atomic per warp at most
  bits = __reduce_or_sync(0xFFFFFFFFu, bits);
  if (bits && (threadIdx.x & 31) == 0) atomicOr(a.err, bits);
}

// Page generation tags: request b reads pages block_tables[b][0 .. used-1];
// each must still carry the tag the request recorded when it mapped it.
struct TagArgs {
  const int32_t* block_tables;
  const uint32_t* table_tags;
  const int32_t* context_lens;
  const uint32_t* page_tags;
  int32_t* status;
  int max_pages, P;
  int64_t num_pages;
};

// One CTA per request; each thread keeps kTagUnroll block-table loads and then
// kTagUnroll tag loads in flight, so a row of up to 8192 entries costs two
// memory round trips.  The CTA writes the request's status itself.
constexpr int kTagThreads = 1024, kTagUnroll = 8;
__global__ void __launch_bounds__(kTagThreads) verify_tags_kernel(const TagArgs a) {
  const int b = blockIdx.x;
  int bad = 0, mismatch = 0;
  int L = a.context_lens[b];
  if (L < 0 || L > a.max_pages * a.P) {
    bad = 1;
    L = L < 0 ? 0 : a.max_pages * a.P;
  }
  const int used = (L + a.P - 1) / a.P;
  const int64_t row = (int64_t)b * a.max_pages;
  for (int base = 0; base < used; base += kTagThreads * kTagUnroll) {
    int page[kTagUnroll];
    uint32_t want[kTagUnroll];
#pragma unroll
    for (int k = 0; k < kTagUnroll; ++k) {
      const int i = base + threadIdx.x + kTagThreads * k;
      page[k] = i < used ? a.block_tables[row + i] : 0;
      want[k] = i < used ? a.table_tags[row + i] : 0;
    }
    uint32_t have[kTagUnroll];
#pragma unroll
    for (int k = 0; k < kTagUnroll; ++k) {
      const int i = base + threadIdx.x + kTagThreads * k;
      const bool in_pool = page[k] >= 0 && page[k] < a.num_pages;
      if (i < used && !in_pool) bad = 1;
      have[k] = (i < used && in_pool) ? a.page_tags[page[k]] : want[k];
    }
#pragma unroll
    for (int k = 0; k < kTagUnroll; ++k) mismatch |= have[k] != want[k];
  }
  bad = __syncthreads_or(bad);
  mismatch = __syncthreads_or(mismatch);
  if (threadIdx.x == 0) a.status[b] = (mismatch ? PFKV_REQ_TAG_MISMATCH : 0) | (bad ? PFKV_REQ_BAD_INDEX : 0);
}

}  // namespace
}  // namespace pfkv

extern "C" int pfkv_validate_tables(const int32_t* block_tables, int max_pages_per_seq,
                                    const int32_t* context_lens, int batch, int page_size,
                                    int64_t num_pages, const int32_t* topk_idx, int topk,
                                    const int64_t* slot_mapping, int num_slots, int32_t* d_err_word,
                                    pfkv_stream_t stream) {
  using namespace pfkv;
  clear_error();
  if (!d_err_word) return fail(PFKV_ERR_INVALID_ARG, "validate_tables: null error word");
  if (batch < 0 || max_pages_per_seq <= 0 || page_size <= 0 || num_pages <= 0 || num_slots < 0 ||
      (topk_idx && topk <= 0))
    return fail(PFKV_ERR_INVALID_ARG, "validate_tables: bad sizes");
  if (batch > 0 && (!block_tables || !context_lens))
    return fail(PFKV_ERR_INVALID_ARG, "validate_tables: null table pointer");
  if (num_slots > 0 && !slot_mapping)
    return fail(PFKV_ERR_INVALID_ARG, "validate_tables: null slot mapping");
  if (!aligned(d_err_word, 4) || (block_tables && !aligned(block_tables, 4)) ||
      (context_lens && !aligned(context_lens, 4)) || (topk_idx && !aligned(topk_idx, 4)) ||
      (num_slots > 0 && !aligned(slot_mapping, 8)))
    return fail(PFKV_ERR_INVALID_ARG, "validate_tables: misaligned pointer");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(d_err_word, 0, sizeof(int32_t), s) != cudaSuccess)
    return check_cuda("validate_tables reset");
  ValidateArgs a;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.topk = topk_idx;
  a.slots = num_slots > 0 ? slot_mapping : nullptr;
  a.err = d_err_word;
  a.B = batch;
  a.max_pages = max_pages_per_seq;
  a.P = page_size;
  a.topk_n = topk_idx ? topk : 0;
  a.num_slots = num_slots;
  a.num_pages = num_pages;
  if (batch == 0 && a.slots == nullptr) return PFKV_OK;
  int span = max_pages_per_seq > a.topk_n ? max_pages_per_seq : a.topk_n;
  if (num_slots > span) span = num_slots;
  int gx = (span + 255) / 256;
  if (gx > 64) gx = 64;
  if (gx < 1) gx = 1;
  dim3 grid(gx, batch + 1);
  validate_kernel<<<grid, 256, 0, s>>>(a);
  return check_cuda("validate_tables launch");
}

extern "C" int pfkv_verify_page_tags(const int32_t* block_tables, const uint32_t* table_tags,
                                     int max_pages_per_seq, const int32_t* context_lens, int batch,
                                     int page_size, const uint32_t* page_tags, int64_t num_pages,
                                     int32_t* request_status, pfkv_stream_t stream) {
  using namespace pfkv;
  clear_error();
  if (batch < 0 || max_pages_per_seq <= 0 || page_size <= 0 || num_pages <= 0)
    return fail(PFKV_ERR_INVALID_ARG, "verify_page_tags: bad sizes");
  if (batch == 0) return PFKV_OK;
  if (!block_tables || !table_tags || !context_lens || !page_tags || !request_status)
    return fail(PFKV_ERR_INVALID_ARG, "verify_page_tags: null pointer");
  if (!aligned(block_tables, 4) || !aligned(table_tags, 4) || !aligned(context_lens, 4) ||
      !aligned(page_tags, 4) || !aligned(request_status, 4))
    return fail(PFKV_ERR_INVALID_ARG, "verify_page_tags: misaligned pointer");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TagArgs a{block_tables, table_tags, context_lens, page_tags, request_status, max_pages_per_seq, page_size, num_pages};
  verify_tags_kernel<<<batch, kTagThreads, 0, s>>>(a);
  return check_cuda("verify_page_tags launch");
}
