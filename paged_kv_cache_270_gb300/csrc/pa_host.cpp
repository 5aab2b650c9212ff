// pa_host.cpp -- host side of the library: pool descriptions and sizing, the
// block allocator (free list + reference counts), copy-on-write preparation
// and error reporting.
//
// The block manager follows the pages' description of PagedAttention as
// virtual memory for the KV cache: a flat pool of fixed 16-token blocks, a
// per-sequence block table, reference-counted sharing of blocks between
// sequences ("Capítulo 8 -- Gestión de caché KV de nueva generación", section
// 8.1), copy-on-write when a sequence starts writing its own tokens into a
// shared block ("PagedAttention y Gestión de KV-Cache", section 3.01), and
// return of every page to the free pool when a request ends or is cancelled
// (same page, section 4.02).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <new>
#include <string>
#include <unordered_map>

#include <nvtx3/nvToolsExt.h>

#include "pa_internal.h"

namespace pa {
// NVTX v3 is header-only: with no tool attached each call is a no-op.
static nvtxDomainHandle_t trace_domain() {
  static nvtxDomainHandle_t d = nvtxDomainCreateA("pagedkv");
  return d;
}

TraceRange::TraceRange(const char* name) {
  nvtxEventAttributes_t e = {};
  e.version = NVTX_VERSION;
  e.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
  e.messageType = NVTX_MESSAGE_TYPE_ASCII;
  e.message.ascii = name;
  nvtxDomainRangePushEx(trace_domain(), &e);
}

TraceRange::~TraceRange() { nvtxDomainRangePop(trace_domain()); }
}  // namespace pa

namespace {
thread_local std::string g_last_error;

int elem_bytes_of(int dtype) {
  switch (dtype) {
    case PA_FP16:
    case PA_BF16:
      return 2;
    case PA_FP8_E4M3:
    case PA_FP8_E4M3_BLOCK:
      return 1;
    default:
      return 0;
  }
}

// Validates everything in a description except num_blocks.
int check_desc_shape(const pa_pool_desc* d) {
  if (!d) return pa::fail(PA_ERR_INVALID, "null pool description");
  if (d->n_layers < 1) return pa::fail(PA_ERR_INVALID, "n_layers must be >= 1 (got %d)", d->n_layers);
  if (d->block_size != PA_BLOCK_SIZE)
    return pa::fail(PA_ERR_UNSUPPORTED, "block_size must be 16 (got %d)", d->block_size);
  if (d->n_kv_heads < 1)
    return pa::fail(PA_ERR_INVALID, "n_kv_heads must be >= 1 (got %d)", d->n_kv_heads);
  if (d->head_dim != 64 && d->head_dim != 128)
    return pa::fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", d->head_dim);
  if (elem_bytes_of(d->kv_dtype) == 0)
    return pa::fail(PA_ERR_UNSUPPORTED, "kv_dtype %d is not a cache type", d->kv_dtype);
  if (d->kv_dtype == PA_FP8_E4M3) {
    if (!(d->k_scale > 0.f) || !std::isfinite(d->k_scale) || !(d->v_scale > 0.f) ||
        !std::isfinite(d->v_scale))
      return pa::fail(PA_ERR_INVALID, "FP8 pools need finite positive k_scale and v_scale");
  }
  return PA_OK;
}

// The kernels address a layer's K or V region as rows of one token of one KV
// head, with the 32-bit signed coordinates of the tensor copies: one layer
// may hold at most this many blocks.
long long max_blocks_per_layer(const pa_pool_desc* d) {
  return 0x7FFFFFFFll / ((long long)d->n_kv_heads * d->block_size);
}

int check_rows(const pa_pool_desc* d) {
  if ((long long)d->num_blocks > max_blocks_per_layer(d))
    return pa::fail(PA_ERR_UNSUPPORTED,
                    "%d blocks x %d kv heads x 16 token rows exceed the 2^31 - 1 rows one layer "
                    "may hold (at most %lld blocks)",
                    d->num_blocks, d->n_kv_heads, max_blocks_per_layer(d));
  return PA_OK;
}

size_t tile_bytes_all_layers(const pa_pool_desc* d) {
  // K + V codes, every layer, one block
  return 2ull * (size_t)d->n_layers * (size_t)d->n_kv_heads * (size_t)d->block_size *
         (size_t)d->head_dim * (size_t)elem_bytes_of(d->kv_dtype);
}

// fp32 scales one block adds to the K and V scale tables (block-scaled FP8 only)
size_t scale_bytes_per_block(const pa_pool_desc* d) {
  return d->kv_dtype == PA_FP8_E4M3_BLOCK ? 2ull * d->n_layers * d->n_kv_heads * sizeof(float) : 0;
}

size_t block_bytes_all_layers(const pa_pool_desc* d) {
  return tile_bytes_all_layers(d) + scale_bytes_per_block(d);
}
}  // namespace

namespace pa {
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int check_pool_layer(const pa_pool* pool, int layer) {
  if (!pool) return fail(PA_ERR_INVALID, "null pool");
  if (layer < 0 || layer >= pool->desc.n_layers)
    return fail(PA_ERR_INVALID, "layer %d outside [0, %d)", layer, pool->desc.n_layers);
  return PA_OK;
}
}  // namespace pa

extern "C" {

int pa_last_error(char* buf, size_t n) {
  if (buf && n) {
    size_t m = g_last_error.size() < n - 1 ? g_last_error.size() : n - 1;
    memcpy(buf, g_last_error.data(), m);
    buf[m] = '\0';
  }
  return PA_OK;
}

int pa_kv_bytes_per_token(int n_layers, int n_kv_heads, int head_dim, int kv_dtype, size_t* bytes) {
  int b = elem_bytes_of(kv_dtype);
  if (!bytes || n_layers < 1 || n_kv_heads < 1 || head_dim < 1 || b == 0)
    return pa::fail(PA_ERR_INVALID, "pa_kv_bytes_per_token: bad argument");
  *bytes = 2ull * (size_t)n_layers * (size_t)n_kv_heads * (size_t)head_dim * (size_t)b;
  return PA_OK;
}

int pa_pool_bytes(const pa_pool_desc* desc, size_t* k_bytes, size_t* v_bytes) {
  int st = check_desc_shape(desc);
  if (st) return st;
  if (desc->num_blocks < 1) return pa::fail(PA_ERR_INVALID, "num_blocks must be >= 1");
  st = check_rows(desc);
  if (st) return st;
  size_t half = tile_bytes_all_layers(desc) / 2 * (size_t)desc->num_blocks;
  half += (scale_bytes_per_block(desc) / 2 * (size_t)desc->num_blocks + 15) / 16 * 16;
  if (k_bytes) *k_bytes = half;
  if (v_bytes) *v_bytes = half;
  return PA_OK;
}

int pa_pool_blocks_for_budget(const pa_pool_desc* desc, size_t budget_bytes, int* num_blocks) {
  int st = check_desc_shape(desc);
  if (st) return st;
  if (!num_blocks) return pa::fail(PA_ERR_INVALID, "null output");
  size_t per = block_bytes_all_layers(desc);
  size_t n = budget_bytes / per;
  // each scale table is rounded up to 16 bytes: drop blocks while that spills over
  auto total = [&](size_t nb) {
    return tile_bytes_all_layers(desc) * nb + 2 * ((scale_bytes_per_block(desc) / 2 * nb + 15) / 16 * 16);
  };
  n = std::min<size_t>(n, (size_t)max_blocks_per_layer(desc));
  while (n > 0 && total(n) > budget_bytes) --n;
  if (n == 0)
    return pa::fail(PA_ERR_NO_MEMORY,
                    "no available memory for the cache blocks: budget %zu B < one block %zu B",
                    budget_bytes, per);
  *num_blocks = n > 0x7FFFFFFF ? 0x7FFFFFFF : (int)n;
  return PA_OK;
}

int pa_pool_create(const pa_pool_desc* desc, void* k_cache, void* v_cache, pa_pool** out) {
  int st = check_desc_shape(desc);
  if (st) return st;
  if (!out) return pa::fail(PA_ERR_INVALID, "null output handle");
  *out = nullptr;
  if (desc->num_blocks < 1) return pa::fail(PA_ERR_NO_MEMORY, "num_blocks must be >= 1");
  st = check_rows(desc);
  if (st) return st;
  if (!k_cache || !v_cache) return pa::fail(PA_ERR_INVALID, "null cache region");
  if (((uintptr_t)k_cache | (uintptr_t)v_cache) & 15u)
    return pa::fail(PA_ERR_INVALID, "cache regions must be 16-byte aligned");
  pa_pool* p = new (std::nothrow) pa_pool;
  if (!p) return pa::fail(PA_ERR_NO_MEMORY, "host allocation failed");
  p->desc = *desc;
  p->k = static_cast<uint8_t*>(k_cache);
  p->v = static_cast<uint8_t*>(v_cache);
  p->elem_bytes = elem_bytes_of(desc->kv_dtype);
  p->tile_bytes = (size_t)desc->block_size * desc->head_dim * p->elem_bytes;
  p->layer_bytes = (size_t)desc->num_blocks * desc->n_kv_heads * p->tile_bytes;
  p->block_scaled = desc->kv_dtype == PA_FP8_E4M3_BLOCK;
  p->scale_offset = p->block_scaled ? (size_t)desc->n_layers * p->layer_bytes : 0;
  try {
    p->refcount.assign(desc->num_blocks, 0);
    p->free_stack.resize(desc->num_blocks);
  } catch (...) {
    delete p;
    return pa::fail(PA_ERR_NO_MEMORY, "host allocation failed");
  }
  // top of the stack is the back: the first pops return 0, 1, 2, ...
  for (int i = 0; i < desc->num_blocks; ++i) p->free_stack[i] = desc->num_blocks - 1 - i;
  *out = p;
  return PA_OK;
}

int pa_pool_destroy(pa_pool* pool) {
  delete pool;
  return PA_OK;
}

int pa_pool_get_desc(const pa_pool* pool, pa_pool_desc* desc) {
  if (!pool || !desc) return pa::fail(PA_ERR_INVALID, "null argument");
  *desc = pool->desc;
  return PA_OK;
}

int pa_block_alloc(pa_pool* pool, int n, int32_t* ids) {
  if (!pool || n < 0 || (n > 0 && !ids)) return pa::fail(PA_ERR_INVALID, "pa_block_alloc: bad argument");
  if ((size_t)n > pool->free_stack.size())
    return pa::fail(PA_ERR_OUT_OF_BLOCKS, "out of cache blocks: need %d, %zu free", n,
                    pool->free_stack.size());
  for (int i = 0; i < n; ++i) {
    int32_t b = pool->free_stack.back();
    pool->free_stack.pop_back();
    pool->refcount[b] = 1;
    ids[i] = b;
  }
  return PA_OK;
}

int pa_block_free(pa_pool* pool, int n, const int32_t* ids) {
  if (!pool || n < 0 || (n > 0 && !ids)) return pa::fail(PA_ERR_INVALID, "pa_block_free: bad argument");
  // validate the whole request first: no change unless every decrement is legal
  std::unordered_map<int32_t, int> count;
  for (int i = 0; i < n; ++i) {
    int32_t b = ids[i];
    if (b < 0 || b >= pool->desc.num_blocks)
      return pa::fail(PA_ERR_INVALID, "free of block %d outside [0, %d)", b, pool->desc.num_blocks);
    if (++count[b] > pool->refcount[b])
      return pa::fail(PA_ERR_INVALID, "free of block %d below refcount 0 (double free)", b);
  }
  for (int i = 0; i < n; ++i) {
    int32_t b = ids[i];
    if (--pool->refcount[b] == 0) pool->free_stack.push_back(b);
  }
  return PA_OK;
}

int pa_block_incref(pa_pool* pool, int n, const int32_t* ids) {
  if (!pool || n < 0 || (n > 0 && !ids)) return pa::fail(PA_ERR_INVALID, "pa_block_incref: bad argument");
  for (int i = 0; i < n; ++i) {
    int32_t b = ids[i];
    if (b < 0 || b >= pool->desc.num_blocks || pool->refcount[b] == 0)
      return pa::fail(PA_ERR_INVALID, "incref of block %d, which is not allocated", b);
  }
  for (int i = 0; i < n; ++i) ++pool->refcount[ids[i]];
  return PA_OK;
}

int pa_block_refcount(const pa_pool* pool, int32_t id, int* refcount) {
  if (!pool || !refcount || id < 0 || id >= pool->desc.num_blocks)
    return pa::fail(PA_ERR_INVALID, "pa_block_refcount: bad argument");
  *refcount = pool->refcount[id];
  return PA_OK;
}

int pa_pool_stats(const pa_pool* pool, int* used, int* free_blocks, int* shared) {
  if (!pool) return pa::fail(PA_ERR_INVALID, "null pool");
  int u = 0, s = 0;
  for (int32_t r : pool->refcount) {
    u += r > 0;
    s += r > 1;
  }
  if (used) *used = u;
  if (free_blocks) *free_blocks = pool->desc.num_blocks - u;
  if (shared) *shared = s;
  return PA_OK;
}

int pa_cow_prepare(pa_pool* pool, int32_t* table_row, int ctx_len, int32_t* src, int32_t* dst,
                   int* n_pairs) {
  if (!pool || !table_row || !src || !dst || !n_pairs || ctx_len < 0)
    return pa::fail(PA_ERR_INVALID, "pa_cow_prepare: bad argument");
  *n_pairs = 0;
  const int B = pool->desc.block_size;
  if (ctx_len % B == 0) return PA_OK;  // the token opens a fresh block
  int32_t old = table_row[ctx_len / B];
  if (old < 0 || old >= pool->desc.num_blocks || pool->refcount[old] == 0)
    return pa::fail(PA_ERR_INVALID, "table entry %d is not an allocated block", old);
  if (pool->refcount[old] <= 1) return PA_OK;  // sole owner writes in place
  int32_t fresh;
  int st = pa_block_alloc(pool, 1, &fresh);
  if (st) return st;
  --pool->refcount[old];  // stays >= 1: still held by the other sharers
  table_row[ctx_len / B] = fresh;
  *src = old;
  *dst = fresh;
  *n_pairs = 1;
  return PA_OK;
}

// ---- prefix caching: block-granular prompt hashing ("Capítulo 8 -- Gestión de
// caché KV de nueva generación", section 8.3)

static uint64_t fnv1a_bytes(uint64_t h, const unsigned char* p, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 1099511628211ull;  // FNV 64-bit prime
  }
  return h;
}

int pa_prefix_hash(const int32_t* tokens, int n_tokens, uint64_t parent, uint64_t* hashes,
                   int* n_blocks) {
  if (n_tokens < 0 || (n_tokens > 0 && !tokens) || !n_blocks)
    return pa::fail(PA_ERR_INVALID, "pa_prefix_hash: bad argument");
  const int nb = n_tokens / PA_BLOCK_SIZE;
  if (nb > 0 && !hashes) return pa::fail(PA_ERR_INVALID, "pa_prefix_hash: null output");
  uint64_t prev = parent;
  for (int j = 0; j < nb; ++j) {
    unsigned char buf[8 + 4 * PA_BLOCK_SIZE];
    for (int b = 0; b < 8; ++b) buf[b] = (unsigned char)(prev >> (8 * b));
    for (int i = 0; i < PA_BLOCK_SIZE; ++i) {
      const uint32_t tkn = (uint32_t)tokens[j * PA_BLOCK_SIZE + i];
      for (int b = 0; b < 4; ++b) buf[8 + 4 * i + b] = (unsigned char)(tkn >> (8 * b));
    }
    prev = fnv1a_bytes(14695981039346656037ull, buf, sizeof buf);  // FNV 64-bit offset basis
    hashes[j] = prev;
  }
  *n_blocks = nb;
  return PA_OK;
}

int pa_prefix_lookup(pa_pool* pool, int n, const uint64_t* hashes, int32_t* ids, int* n_hit) {
  if (!pool || n < 0 || (n > 0 && (!hashes || !ids)) || !n_hit)
    return pa::fail(PA_ERR_INVALID, "pa_prefix_lookup: bad argument");
  int hit = 0;
  pool->prefix_lookups += n;
  const uint64_t tick = ++pool->prefix_tick;
  for (; hit < n; ++hit) {
    auto it = pool->prefix.find(hashes[hit]);
    if (it == pool->prefix.end()) break;
    it->second.last_use = tick;
    ids[hit] = it->second.block;
    ++pool->refcount[it->second.block];
  }
  pool->prefix_hits += hit;
  *n_hit = hit;
  return PA_OK;
}

int pa_prefix_register(pa_pool* pool, int n, const uint64_t* hashes, const int32_t* ids) {
  if (!pool || n < 0 || (n > 0 && (!hashes || !ids)))
    return pa::fail(PA_ERR_INVALID, "pa_prefix_register: bad argument");
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= pool->desc.num_blocks || pool->refcount[ids[i]] == 0)
      return pa::fail(PA_ERR_INVALID, "register of block %d, which is not allocated", ids[i]);
  const uint64_t tick = ++pool->prefix_tick;
  for (int i = 0; i < n; ++i) {
    if (pool->prefix.count(hashes[i])) continue;
    pool->prefix[hashes[i]] = pa_pool::prefix_entry{ids[i], tick};
    ++pool->refcount[ids[i]];
  }
  return PA_OK;
}

int pa_prefix_evict(pa_pool* pool, int max_blocks, int* n_evicted) {
  if (!pool || max_blocks < 0 || !n_evicted)
    return pa::fail(PA_ERR_INVALID, "pa_prefix_evict: bad argument");
  // candidates: entries only the cache references, least recently used first
  // (ties: lower block id first)
  std::vector<std::pair<std::pair<uint64_t, int32_t>, uint64_t>> cand;
  for (const auto& kv : pool->prefix)
    if (pool->refcount[kv.second.block] == 1)
      cand.push_back({{kv.second.last_use, kv.second.block}, kv.first});
  std::sort(cand.begin(), cand.end());
  int ev = 0;
  for (const auto& c : cand) {
    if (ev >= max_blocks) break;
    const int32_t b = c.first.second;
    pool->prefix.erase(c.second);
    pool->refcount[b] = 0;
    pool->free_stack.push_back(b);
    ++ev;
  }
  *n_evicted = ev;
  return PA_OK;
}

int pa_prefix_stats(const pa_pool* pool, int* entries, long long* lookups, long long* hits) {
  if (!pool) return pa::fail(PA_ERR_INVALID, "null pool");
  if (entries) *entries = (int)pool->prefix.size();
  if (lookups) *lookups = pool->prefix_lookups;
  if (hits) *hits = pool->prefix_hits;
  return PA_OK;
}

}  // extern "C"
