// pa_internal.h -- library-internal declarations shared by the host and CUDA
// translation units (not part of the public ABI).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <unordered_map>
#include <vector>

#include "pa.h"  // include/ is on the include path

// Opaque storage for one CUtensorMap (128 bytes, 64-byte aligned).
struct alignas(64) pa_tmap_blob {
  unsigned char bytes[128];
};

struct pa_pool {
  pa_pool_desc desc;
  uint8_t* k;                     // device, all layers
  uint8_t* v;                     // device, all layers
  int elem_bytes;                 // 1 (FP8) or 2
  size_t tile_bytes;              // one (block, kv head) tile: block_size * head_dim * elem_bytes
  size_t layer_bytes;             // one layer of K (or V): num_blocks * n_kv_heads * tile_bytes
  // PA_FP8_E4M3_BLOCK: byte offset, in the K and in the V region, of the fp32
  // scale table [n_layers][num_blocks][n_kv_heads] (= n_layers * layer_bytes); 0 otherwise.
  bool block_scaled = false;
  size_t scale_offset = 0;
  std::vector<int32_t> refcount;  // per block
  std::vector<int32_t> free_stack;  // top = back()
  // TMA descriptors of each layer's K and V regions ([2 * layer + {0: K, 1: V}]),
  // encoded on first use by pa_decode.
  std::vector<pa_tmap_blob> tmaps;
  std::vector<char> tmap_ready;  // per layer
  // 16-bit pools: maps whose box is one 64-element half of each row (the
  // tensor-core prefill), encoded on first use the same way
  std::vector<pa_tmap_blob> tmaps_half;
  std::vector<char> tmap_half_ready;
  // Prefix cache: chain hash of a full block -> the block holding its K/V.
  // The cache owns one reference to each block it maps.
  struct prefix_entry {
    int32_t block;
    uint64_t last_use;  // tick of the last lookup or registration
  };
  std::unordered_map<uint64_t, prefix_entry> prefix;
  uint64_t prefix_tick = 0;
  long long prefix_lookups = 0;  // blocks asked for
  long long prefix_hits = 0;     // blocks found
};

namespace pa {

// An NVTX range (domain "pagedkv") around one library call: it shows in a
// profiler's timeline with the kernels the call launched.  NVTX does nothing
// unless a profiling tool is attached to the process.
struct TraceRange {
  explicit TraceRange(const char* name);
  ~TraceRange();
};

// Records `msg` as the calling thread's last error and returns `code`.
int fail(int code, const char* fmt, ...);

// Address of the per-device error word (current device); nullptr on failure
// (the error is then recorded and PA_ERR_CUDA should be returned).
unsigned int* device_error_word();

int check_pool_layer(const pa_pool* pool, int layer);

// The K and V scale tables of `layer` of a block-scaled pool: fp32 [num_blocks][n_kv_heads].
inline float* layer_scales(const pa_pool* p, uint8_t* region, int layer) {
  return reinterpret_cast<float*>(region + p->scale_offset) +
         (size_t)layer * p->desc.num_blocks * p->desc.n_kv_heads;
}

}  // namespace pa

struct CUtensorMap_st;
namespace pa {
// TMA descriptors (CUtensorMap) of one layer's K and V regions, encoded on
// first use and kept in the pool; rows of one token of one kv head, a box is
// one 16-token tile, 128-byte swizzled when a row is 128 or 256 bytes.
int layer_maps(pa_pool* pool, int layer, const CUtensorMap_st** tk, const CUtensorMap_st** tv);
// The same regions for 16-bit pools as rows of 256 bytes with a 128-byte box,
// so one page is loaded as two 64-element halves (x = 0 and x = 128 bytes).
int layer_half_maps(pa_pool* pool, int layer, const CUtensorMap_st** tk, const CUtensorMap_st** tv);

// Set the pipeline wait limit of each translation unit's kernels (see
// pa_set_pipeline_wait_limit_ns); they return a cudaError_t value.
int decode_set_wait_limit(unsigned long long ns);
int prefill_set_wait_limit(unsigned long long ns);
int prefill_tc_set_wait_limit(unsigned long long ns);

// Chunked prefill on the tcgen05 tensor cores, for the shapes it covers
// (head_dim 128, 1, 2, 4 or 8 query heads per KV head; FP8 or bfloat16 pools with bf16 or
// fp32 output, binary16 pools with fp16 or fp32 output); the arguments are
// those of pa_prefill, already validated.
bool prefill_tc_supported(const pa_pool* pool, int n_q_heads, int out_dtype);
int prefill_tc(pa_pool* pool, int layer, void* out, int out_dtype, const void* q, const int32_t* q_start,
               const int32_t* tables, int max_blocks, const int32_t* ctx, int S, int n_q_heads,
               int max_chunk, float softmax_scale, unsigned int* err, struct CUstream_st* st);

}  // namespace pa
