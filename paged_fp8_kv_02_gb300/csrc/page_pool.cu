// page_pool.cu -- host-side page pool and prefix cache for the paged KV cache.
//
// Explainer page (KV cache explainer, "PagedAttention の 2 つの原語"): the cache
// is a pool of fixed-size blocks plus a per-request block table mapping
// logical block numbers to physical ones; allocating is popping a block number
// off a free list and freeing is pushing it back, O(1) whatever the
// fragmentation and without any device allocation; blocks can be shared, which
// is what the prefix cache stands on.  "Prefix Cache" section ("原理：ブロック
// 単位のハッシュ"): every full block is identified by a hash of its tokens and
// of its parent block's hash, so a block's hash fingerprints everything before
// it; a lookup walks the blocks of a prompt in order and stops at the first
// miss, which floors the reused length to whole blocks.
//
// Here the pool also keeps, per page, a reference count (a shared page is freed
// when its last holder releases it) and a generation tag that changes each time
// the page is handed out, which pfkv_verify_page_tags checks before decode.
// The block hash is 64-bit FNV-1a over the parent hash (8 bytes, little
// endian) followed by the block's token ids (4 bytes each, little endian); the
// root block's parent is 0.  A hit trusts the 64-bit hash.  A page whose last
// reference is released leaves the prefix table at once (no cache of
// unreferenced blocks).  Not thread-safe: one pool per scheduler thread.
#include <stdint.h>

#include <new>
#include <unordered_map>
#include <vector>

#include "pfkv_internal.h"

struct pfkv_page_pool {
  int64_t num_pages = 0;
  int page_size = 0;
  std::vector<int32_t> free_list;   // stack of free page ids
  std::vector<int32_t> refcount;    // holders of each page
  std::vector<uint32_t> tag;        // generation: changes at every hand-out
  std::vector<uint64_t> page_hash;  // prefix hash a page is registered under
  std::vector<uint8_t> registered;  // page_hash[p] is in the prefix table
  std::unordered_map<uint64_t, int32_t> prefix;  // block hash -> page
};

namespace {

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

uint64_t fnv1a(uint64_t h, const uint8_t* bytes, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    h ^= bytes[i];
    h *= kFnvPrime;
  }
  return h;
}

uint64_t block_hash(uint64_t parent, const int32_t* tokens, int n) {
  uint8_t buf[8];
  for (int i = 0; i < 8; ++i) buf[i] = (uint8_t)(parent >> (8 * i));
  uint64_t h = fnv1a(kFnvOffset, buf, 8);
  for (int t = 0; t < n; ++t) {
    const uint32_t v = (uint32_t)tokens[t];
    for (int i = 0; i < 4; ++i) buf[i] = (uint8_t)(v >> (8 * i));
    h = fnv1a(h, buf, 4);
  }
  return h;
}

// Pop a free page: O(1).  Its tag moves on so that stale block-table entries
// pointing at it no longer verify.
int32_t take_page(pfkv_page_pool* p) {
  const int32_t page = p->free_list.back();
  p->free_list.pop_back();
  p->refcount[page] = 1;
  p->tag[page] += 1;
  return page;
}

void drop_ref(pfkv_page_pool* p, int32_t page) {
  if (--p->refcount[page] > 0) return;
  if (p->registered[page]) {
    auto it = p->prefix.find(p->page_hash[page]);
    if (it != p->prefix.end() && it->second == page) p->prefix.erase(it);
    p->registered[page] = 0;
  }
  p->free_list.push_back(page);
}

}  // namespace

extern "C" {

uint64_t pfkv_block_hash(uint64_t parent, const int32_t* tokens, int n) {
  if (n < 0 || (n > 0 && tokens == nullptr)) return 0;
  return block_hash(parent, tokens, n);
}

pfkv_page_pool* pfkv_pool_create(int64_t num_pages, int page_size) {
  pfkv::clear_error();
  if (num_pages <= 0 || num_pages > INT32_MAX || page_size <= 0) {
    pfkv::fail(PFKV_ERR_INVALID_ARG, "pool_create: bad sizes");
    return nullptr;
  }
  pfkv_page_pool* p = new (std::nothrow) pfkv_page_pool;
  if (p == nullptr) {
    pfkv::fail(PFKV_ERR_INVALID_ARG, "pool_create: out of host memory");
    return nullptr;
  }
  try {
    p->num_pages = num_pages;
    p->page_size = page_size;
    p->free_list.resize((size_t)num_pages);
    for (int64_t i = 0; i < num_pages; ++i) p->free_list[(size_t)i] = (int32_t)(num_pages - 1 - i);  // pops 0, 1, ...
    p->refcount.assign((size_t)num_pages, 0);
    p->tag.assign((size_t)num_pages, 0);
    p->page_hash.assign((size_t)num_pages, 0);
    p->registered.assign((size_t)num_pages, 0);
  } catch (...) {
    delete p;
    pfkv::fail(PFKV_ERR_INVALID_ARG, "pool_create: out of host memory");
    return nullptr;
  }
  return p;
}

void pfkv_pool_destroy(pfkv_page_pool* pool) { delete pool; }

int64_t pfkv_pool_num_free(const pfkv_page_pool* pool) {
  return pool ? (int64_t)pool->free_list.size() : -1;
}

int pfkv_pool_refcount(const pfkv_page_pool* pool, int32_t page) {
  if (pool == nullptr || page < 0 || page >= pool->num_pages) return -1;
  return pool->refcount[page];
}

int pfkv_pool_page_tags(const pfkv_page_pool* pool, uint32_t* tags_out) {
  pfkv::clear_error();
  if (pool == nullptr || tags_out == nullptr) return pfkv::fail(PFKV_ERR_INVALID_ARG, "pool_page_tags: null pointer");
  for (int64_t i = 0; i < pool->num_pages; ++i) tags_out[i] = pool->tag[(size_t)i];
  return PFKV_OK;
}

int pfkv_pool_map_request(pfkv_page_pool* pool, const int32_t* tokens, int n_tokens, int32_t* block_table_row,
                          uint32_t* table_tags, int max_pages, int* cached_tokens) {
  pfkv::clear_error();
  if (pool == nullptr || block_table_row == nullptr || table_tags == nullptr || cached_tokens == nullptr ||
      (n_tokens > 0 && tokens == nullptr))
    return pfkv::fail(PFKV_ERR_INVALID_ARG, "pool_map_request: null pointer");
  if (n_tokens < 0 || max_pages <= 0) return pfkv::fail(PFKV_ERR_INVALID_ARG, "pool_map_request: bad sizes");
  const int P = pool->page_size;
  const int n_pages = (n_tokens + P - 1) / P;
  const int n_full = n_tokens / P;
  if (n_pages > max_pages)
    return pfkv::fail(PFKV_ERR_INVALID_ARG, "pool_map_request: %d pages needed, row holds %d", n_pages, max_pages);
  // Walk the full blocks while they hit; every later block gets a fresh page.
  uint64_t h = 0;
  int hits = 0;
  std::vector<uint64_t> hashes((size_t)n_full);
  for (int i = 0; i < n_full; ++i) {
    h = block_hash(h, tokens + (int64_t)i * P, P);
    hashes[(size_t)i] = h;
  }
  for (; hits < n_full; ++hits) {
    auto it = pool->prefix.find(hashes[(size_t)hits]);
    if (it == pool->prefix.end()) break;
  }
  if ((int64_t)(n_pages - hits) > (int64_t)pool->free_list.size())
    return pfkv::fail(PFKV_ERR_NO_PAGES, "pool_map_request: %d free pages needed, %lld left", n_pages - hits,
                      (long long)pool->free_list.size());
  for (int i = 0; i < hits; ++i) {
    const int32_t page = pool->prefix.find(hashes[(size_t)i])->second;
    pool->refcount[page] += 1;
    block_table_row[i] = page;
    table_tags[i] = pool->tag[page];
  }
  for (int i = hits; i < n_pages; ++i) {
    const int32_t page = take_page(pool);
    block_table_row[i] = page;
    table_tags[i] = pool->tag[page];
    if (i < n_full) {  // a full block: later prompts with the same prefix reuse it
      pool->prefix[hashes[(size_t)i]] = page;
      pool->page_hash[page] = hashes[(size_t)i];
      pool->registered[page] = 1;
    }
  }
  for (int i = n_pages; i < max_pages; ++i) {
    block_table_row[i] = -1;
    table_tags[i] = 0;
  }
  *cached_tokens = hits * P;
  return PFKV_OK;
}

int pfkv_pool_release(pfkv_page_pool* pool, const int32_t* block_table_row, int n_pages) {
  pfkv::clear_error();
  if (pool == nullptr || (n_pages > 0 && block_table_row == nullptr))
    return pfkv::fail(PFKV_ERR_INVALID_ARG, "pool_release: null pointer");
  // Each entry drops one reference, so a page listed k times must hold k:
  // take the references tentatively, put them back, and fail on the first
  // entry that finds none left (the pool is then unchanged).
  int i = 0;
  for (; i < n_pages; ++i) {
    const int32_t page = block_table_row[i];
    if (page < 0 || page >= pool->num_pages || pool->refcount[page] <= 0) break;
    --pool->refcount[page];
  }
  for (int j = 0; j < i; ++j) ++pool->refcount[block_table_row[j]];
  if (i < n_pages)
    return pfkv::fail(PFKV_ERR_INVALID_ARG, "pool_release: page %d (entry %d) is not held", block_table_row[i], i);
  for (int k = 0; k < n_pages; ++k) drop_ref(pool, block_table_row[k]);
  return PFKV_OK;
}

int pfkv_slots_from_table(const int32_t* block_table_row, int max_pages, int page_size, int first_token,
                          int n_tokens, int64_t* slots_out) {
  pfkv::clear_error();
  if (block_table_row == nullptr || (n_tokens > 0 && slots_out == nullptr))
    return pfkv::fail(PFKV_ERR_INVALID_ARG, "slots_from_table: null pointer");
  if (page_size <= 0 || first_token < 0 || n_tokens < 0 || (int64_t)first_token + n_tokens > (int64_t)max_pages * page_size)
    return pfkv::fail(PFKV_ERR_INVALID_ARG, "slots_from_table: bad range");
  for (int k = 0; k < n_tokens; ++k) {
    const int t = first_token + k;
    const int32_t page = block_table_row[t / page_size];
    if (page < 0) return pfkv::fail(PFKV_ERR_INVALID_ARG, "slots_from_table: token %d has no page", t);
    slots_out[k] = (int64_t)page * page_size + t % page_size;
  }
  return PFKV_OK;
}

}  // extern "C"
