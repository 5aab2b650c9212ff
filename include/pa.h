/*
 * pa.h -- C ABI of the paged KV-cache decode library (GB300, sm_103a).
 *
 * The KV cache lives in a flat physical pool of fixed-size blocks of 16 tokens;
 * each sequence addresses it through a block table mapping logical block j to
 * a physical block id, and the attention kernel gathers keys and values by
 * that indirection instead of slicing a contiguous slab ("Capítulo 8 --
 * Gestión de caché KV de nueva generación", section 8.1; "PagedAttention y
 * Gestión de KV-Cache", section 2 figure).  The cache may hold FP8 E4M3 codes
 * with a static per-tensor scale ("Optimización de KV Cache con
 * PagedAttention y Cuantización FP8 para Contextos Largos (128K)", sections 4
 * and 8).  Blocks are reference counted so sequences can share a prefix, with
 * copy-on-write before a sequence appends into a shared block ("PagedAttention
 * y Gestión de KV-Cache", sections 3.01 and 3.02; "KV Cache y PagedAttention",
 * "Cómo PagedAttention soluciona esto").
 *
 * Conventions, for every function below:
 *  - Returns a status: PA_OK (0) or one of the PA_ERR_* codes.  Nothing
 *    throws across the ABI.  pa_last_error() gives the calling thread's last
 *    message.
 *  - Device pointers are owned by the caller.  The library never allocates or
 *    frees device memory.  Host arrays passed in are read (or written, where
 *    stated) during the call only.
 *  - Functions taking a `stream` (a cudaStream_t passed as void*; NULL is the
 *    legacy default stream) only enqueue work: they are asynchronous and do
 *    not synchronise.  Problems found by a kernel (an out-of-range block id or
 *    slot, a context longer than its table, a pipeline wait that timed out)
 *    are recorded in a per-device error word; read it with
 *    pa_get_device_error().  Kernels never trap: they skip the bad access.
 *  - A pool handle is not thread-safe: use it from one thread at a time.
 *  - Every device buffer must be 16-byte aligned.
 *
 * Pool layout in device memory (per layer l, for K and for V separately):
 *   [num_blocks][n_kv_heads][block_size][head_dim] elements, layer l at byte
 *   offset l * num_blocks * n_kv_heads * block_size * head_dim * elem_bytes.
 *   One (block, kv head) tile of block_size * head_dim elements is contiguous.
 *   A PA_FP8_E4M3_BLOCK region continues, right after the tiles of its last
 *   layer, with its scale table: fp32 [n_layers][num_blocks][n_kv_heads], the
 *   scale of each (layer, block, kv head) tile of that region.
 */
#ifndef PAGED_KV_PA_H
#define PAGED_KV_PA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define PA_OK 0
#define PA_ERR_INVALID 1       /* bad argument or request (nothing changed) */
#define PA_ERR_UNSUPPORTED 2   /* valid but not implemented (e.g. head_dim 96) */
#define PA_ERR_OUT_OF_BLOCKS 3 /* the free list cannot satisfy an allocation */
#define PA_ERR_NO_MEMORY 4     /* a budget that holds no block at all */
#define PA_ERR_CUDA 5          /* a CUDA runtime call failed */
#define PA_ERR_BOUNDS 6        /* a kernel met an out-of-range id, slot or length */
#define PA_ERR_TIMEOUT 7       /* a kernel pipeline wait gave up (bounded spin) */

/* ---- element types ---- */
#define PA_FP16 0     /* IEEE binary16 */
#define PA_BF16 1     /* bfloat16 */
#define PA_FP8_E4M3 2 /* OCP FP8 E4M3FN codes, value = decode(code) * scale */
#define PA_FP32 3     /* IEEE binary32 (decode output only: the fp32 check mode) */
/* OCP FP8 E4M3FN codes with a dynamic scale per (block, kv head) tile, for K
 * and for V: value = decode(code) * s, s = fl32(MaxAbs / 448) of the values
 * the tile holds, kept in the region's scale table ("Optimización de KV Cache
 * ...", section 8, dynamic scaling: the MaxAbs of each block is computed at
 * inference time).  s = 0 marks an all-zero tile.  See pa_reshape_and_cache. */
#define PA_FP8_E4M3_BLOCK 4

#define PA_BLOCK_SIZE 16

/* Description of a KV pool.
 *   n_layers    layers held by the pool (each layer has its own K and V region)
 *   num_blocks  physical blocks per layer (>= 1)
 *   block_size  tokens per block; must be 16
 *   n_kv_heads  KV heads (>= 1)
 *   head_dim    64 or 128
 *   kv_dtype    PA_FP16, PA_BF16, PA_FP8_E4M3 or PA_FP8_E4M3_BLOCK.  FP16
 *               pools take binary16 q/k/v; the others take bfloat16 q/k/v.
 *   k_scale, v_scale  PA_FP8_E4M3 only: static per-tensor scales (> 0,
 *               finite); a code c stands for decode(c) * scale.  Ignored for
 *               the other types. */
typedef struct pa_pool_desc {
  int n_layers;
  int num_blocks;
  int block_size;
  int n_kv_heads;
  int head_dim;
  int kv_dtype;
  float k_scale;
  float v_scale;
} pa_pool_desc;

typedef struct pa_pool pa_pool;

/* Copies the calling thread's last error message into buf (NUL-terminated,
 * truncated to n bytes).  Returns PA_OK. */
PA_API int pa_last_error(char* buf, size_t n);

/* KV bytes per token of a model: 2 * n_layers * n_kv_heads * head_dim *
 * bytes(kv_dtype) -- one K and one V vector per KV head per layer
 * ("Optimización de KV Cache ...", section 2, worked example 327,680 bytes for
 * 80 layers, 8 KV heads, head dim 128, FP16; FP8 halves it, section 4). */
PA_API int pa_kv_bytes_per_token(int n_layers, int n_kv_heads, int head_dim, int kv_dtype,
                          size_t* bytes);

/* Bytes of device memory the caller must provide for the K region and for the
 * V region of a pool described by *desc (all layers; for PA_FP8_E4M3_BLOCK the
 * scale table included, the total rounded up to a multiple of 16).
 * PA_ERR_UNSUPPORTED if one layer would hold more than 2^31 - 1 token rows
 * (num_blocks * n_kv_heads * 16): the kernels address a layer's region with
 * the 32-bit signed row coordinates of the tensor copies. */
PA_API int pa_pool_bytes(const pa_pool_desc* desc, size_t* k_bytes, size_t* v_bytes);

/* Largest num_blocks whose K + V regions (tiles and, for PA_FP8_E4M3_BLOCK,
 * 2 * n_layers * n_kv_heads fp32 scales per block) fit in budget_bytes
 * (desc->num_blocks is ignored), and at most the 2^31 - 1 token rows per layer that
 * pa_pool_bytes allows.  PA_ERR_NO_MEMORY if not even one block fits -- the "no
 * available memory for the cache blocks" start-up failure ("Optimización de KV
 * Cache ...", section 6.1). */
PA_API int pa_pool_blocks_for_budget(const pa_pool_desc* desc, size_t budget_bytes, int* num_blocks);

/* Creates a pool over caller-owned device regions k_cache and v_cache (each at
 * least the pa_pool_bytes size, 16-byte aligned).  The host allocator starts
 * with every block free; its LIFO free list hands out 0, 1, 2, ... first.
 * The pool does not own the device memory.  The same limit of 2^31 - 1 token
 * rows per layer as pa_pool_bytes (PA_ERR_UNSUPPORTED). */
PA_API int pa_pool_create(const pa_pool_desc* desc, void* k_cache, void* v_cache, pa_pool** out);

/* Destroys the host state of a pool (device memory is untouched). NULL is OK. */
PA_API int pa_pool_destroy(pa_pool* pool);

/* Copies the pool's description into *desc. */
PA_API int pa_pool_get_desc(const pa_pool* pool, pa_pool_desc* desc);

/* ---- host block allocator ("Capítulo 8 ...", section 8.1: free list and
 * reference-counted sharing; "PagedAttention y Gestión de KV-Cache",
 * section 4.02: pages return to the free pool when a request ends) ---- */

/* Allocates n blocks (refcount 1 each) into ids[0..n).  All or nothing:
 * PA_ERR_OUT_OF_BLOCKS leaves the pool unchanged.  Freed blocks are reused
 * first (LIFO). */
PA_API int pa_block_alloc(pa_pool* pool, int n, int32_t* ids);

/* Drops one reference from each of ids[0..n) (an id may repeat); a block whose
 * count reaches 0 goes back on the free list, in argument order.
 * PA_ERR_INVALID (and no change at all) if any id is out of range or would go
 * below zero -- a double free. */
PA_API int pa_block_free(pa_pool* pool, int n, const int32_t* ids);

/* Adds one reference to each of ids[0..n) (sharing a block with another
 * sequence).  PA_ERR_INVALID (no change) if any id is free or out of range. */
PA_API int pa_block_incref(pa_pool* pool, int n, const int32_t* ids);

/* Current reference count of block id (0 = free). */
PA_API int pa_block_refcount(const pa_pool* pool, int32_t id, int* refcount);

/* Blocks in use (refcount > 0), free, and shared (refcount > 1); any output
 * pointer may be NULL.  used / num_blocks is the cache usage factor a serving
 * monitor watches ("Optimización de KV Cache ...", section 7). */
PA_API int pa_pool_stats(const pa_pool* pool, int* used, int* free_blocks, int* shared);

/* Copy-on-write preparation for appending token number ctx_len (0-based) to a
 * sequence whose block table is table_row (host array, at least
 * ctx_len / 16 + 1 entries).  If the token falls inside an existing block
 * (ctx_len % 16 != 0) whose refcount is above 1, a new block is allocated, the
 * shared one loses a reference, table_row[ctx_len / 16] is rewritten to the
 * new id, and (*src, *dst) = (old, new) with *n_pairs = 1: the caller then
 * copies the block contents with pa_copy_blocks before writing the token.
 * Otherwise *n_pairs = 0 and nothing changes (a token that opens a new block
 * needs pa_block_alloc, not a copy).  PA_ERR_OUT_OF_BLOCKS if no block is
 * free (no change). */
PA_API int pa_cow_prepare(pa_pool* pool, int32_t* table_row, int ctx_len, int32_t* src, int32_t* dst,
                   int* n_pairs);

/* ---- prefix caching ("Capítulo 8 ...", section 8.3: hash the prompt in
 * block-size chunks; a request whose leading blocks are already cached points
 * its block table at them and skips their prefill; new full blocks are
 * registered after their prefill) ----
 * A block's key is a chain hash: h_j = FNV-1a-64 over the 8 little-endian bytes
 * of h_{j-1} followed by the 16 token ids of block j (4 little-endian bytes
 * each), with h_{-1} = `parent` (0 for the start of a prompt).  Only full
 * blocks are hashed and cached.  Two different prefixes with equal 64-bit
 * hashes would share a block (not checked). */

/* Chain hashes of the floor(n_tokens / 16) full blocks of tokens[0..n_tokens),
 * written to hashes[]; *n_blocks receives their count.  Host only. */
PA_API int pa_prefix_hash(const int32_t* tokens, int n_tokens, uint64_t parent, uint64_t* hashes,
                          int* n_blocks);

/* Looks up hashes[0..n) in order and stops at the first miss.  For each hit
 * (the leading *n_hit of them) ids[i] receives the cached block, which gains a
 * reference for the caller's table.  Entries hit become the most recently
 * used. */
PA_API int pa_prefix_lookup(pa_pool* pool, int n, const uint64_t* hashes, int32_t* ids, int* n_hit);

/* Registers full blocks ids[i] (allocated, holding the K/V of the block whose
 * chain hash is hashes[i]).  The cache takes one reference to each block it
 * adds; hashes already cached are left as they are.  PA_ERR_INVALID (no change)
 * if an id is not an allocated block. */
PA_API int pa_prefix_register(pa_pool* pool, int n, const uint64_t* hashes, const int32_t* ids);

/* Evicts up to max_blocks cached entries whose block no request references
 * (refcount 1: only the cache), least recently used first; their blocks go back
 * on the free list.  *n_evicted receives the count. */
PA_API int pa_prefix_evict(pa_pool* pool, int max_blocks, int* n_evicted);

/* Cached entries, and the blocks looked up / found since the pool was made;
 * any output pointer may be NULL. */
PA_API int pa_prefix_stats(const pa_pool* pool, int* entries, long long* lookups, long long* hits);

/* ---- device operations ---- */

/* For each pair p < n_pairs of pairs_dev (device int32 [n_pairs][2] =
 * (src, dst)), copies the K and V tiles of every KV head of block src into
 * block dst, in layer `layer` (the device half of copy-on-write).  Pairs with
 * an id outside [0, num_blocks) are skipped and set PA_ERR_BOUNDS in the device
 * error word.  Destinations must be distinct and no destination may also be a
 * source in the same call.  PA_FP8_E4M3_BLOCK pools copy the tiles' scales
 * with them. */
PA_API int pa_copy_blocks(pa_pool* pool, int layer, const int32_t* pairs_dev, int n_pairs, void* stream);

/* ---- page swap to host memory ("KV Cache y PagedAttention", "Cómo
 * PagedAttention soluciona esto": under memory pressure the system moves small
 * pages to the CPU instead of whole sequences; "PagedAttention y Gestión de
 * KV-Cache", KV-cache offloading to system RAM) ----
 * A swapped block is the K and V of every kv head of every layer:
 * pa_swap_block_bytes per block, laid out in the host buffer as
 * [block][layer][K | V][n_kv_heads][block_size][head_dim] elements; for
 * PA_FP8_E4M3_BLOCK each block's record continues with its scales, fp32
 * [layer][K | V][n_kv_heads], then zero bytes up to a multiple of 16.  The host
 * buffer must be page-locked and device-accessible (cudaHostAlloc /
 * cudaMallocHost, or cudaHostRegister'ed memory); the GPU reads or writes it
 * directly over the CPU-GPU link. */

/* Bytes one block occupies in a swap buffer. */
PA_API int pa_swap_block_bytes(const pa_pool* pool, size_t* bytes);

/* Copies blocks ids_dev[0..n) (device int32) into host_buf, block i at offset
 * i * pa_swap_block_bytes.  The blocks' refcounts are not touched: free them
 * with pa_block_free once the copy is ordered before any reuse (work later on
 * the same stream is).  Out-of-range ids are skipped and set PA_ERR_BOUNDS. */
PA_API int pa_swap_out(pa_pool* pool, int n, const int32_t* ids_dev, void* host_buf, void* stream);

/* Copies host_buf (as written by pa_swap_out) back into blocks ids_dev[0..n),
 * e.g. freshly allocated ones whose ids then replace the old ones in the block
 * table.  Out-of-range ids are skipped and set PA_ERR_BOUNDS. */
PA_API int pa_swap_in(pa_pool* pool, int n, const int32_t* ids_dev, const void* host_buf,
                      void* stream);

/* Writes T new tokens into their slots of layer `layer` (scatter through the
 * slot mapping; pages are filled on demand, "Optimización de KV Cache ...",
 * section 3).
 *   k, v              device [T][n_kv_heads][head_dim], binary16 for FP16
 *                     pools, bfloat16 for BF16 and FP8 pools
 *   slot_mapping_dev  device int64 [T]: slot = block * 16 + offset, or negative
 *                     to skip the token; a slot >= num_blocks * 16 is skipped
 *                     and sets PA_ERR_BOUNDS in the device error word
 * FP8 pools store code = E4M3(round-to-nearest-even, saturating to +-448) of
 * the IEEE fp32 quotient x / scale ("Optimización de KV Cache ...", sections 4
 * and 8, static calibration).  16-bit pools store x unchanged.  Two tokens with
 * the same slot in one call race.
 *
 * PA_FP8_E4M3_BLOCK pools (same page, section 8, dynamic scaling) take the
 * tokens in runs: a token and the tokens right after it in slot_mapping whose
 * slots follow it within the same block.  For each run and kv head, separately
 * for K and V, with m = max |x| over the run and s_run = fl32(m / 448):
 *   - a run starting at offset 0 of its block starts the tile afresh: s = s_run;
 *   - a run starting at offset o > 0 appends: s = max(s_old, s_run); if s grew,
 *     every code c of rows 0 .. o-1 is re-encoded as
 *     E4M3(fl32(fl32(decode(c) * s_old) / s)) (the originals are not kept);
 *   - the run's values are stored as E4M3(fl32(x / s)), code 0 when s = 0;
 *   - s goes to the scale table.
 * The tokens one call writes into one block must form a single run (a
 * sequence's new tokens in order do); two runs into one block in one call
 * race.  A tile must be started at offset 0 before it is appended to. */
PA_API int pa_reshape_and_cache(pa_pool* pool, int layer, const void* k, const void* v,
                         const int64_t* slot_mapping_dev, int T, void* stream);

/* num_splits value that asks pa_decode for the balanced schedule (batches of
 * at most 4096 sequences, else PA_ERR_UNSUPPORTED): one CTA per resident slot
 * of the GPU, four per SM (the kernel's shared memory keeps a fifth off); the
 * (sequence, kv head) pairs, taken in (sequence, kv head, page) order, are cut
 * into contiguous ranges of equal cost, one per CTA, from the context lengths
 * on the device: a pair of n pages costs n plus a fixed 12 pages (FP8 pools;
 * 6 for 16-bit pools), what finishing a pair costs a CTA.  Every CTA thus
 * streams about as long whatever the mix of lengths, and streams from one
 * pair to the next without draining its pipeline.  A pair whose pages span
 * several CTAs is merged by a second kernel.  For batches whose lengths differ
 * by orders of magnitude, which the automatic split count (sized from the
 * table width) serves badly. */
#define PA_SPLITS_BALANCED (-1)

/* Number of splits pa_decode uses along each sequence's pages for this batch
 * shape when num_splits = 0 (auto): enough (sequence, KV head, split) work
 * units to fill the GPU, each split still covering several pages (every
 * sequence is taken as max_blocks_per_seq pages long: the lengths live on the
 * device).  When that count s is at least 2 and its CTAs take more than one
 * wave of the GPU, the automatic layout is guided instead: min(2 s, 8) splits
 * whose shares of the table fall geometrically (ratio 0.55), handed out split
 * by split (every sequence's first split before any second one), so the CTAs
 * that run last, as the grid drains, are short; this returns that count.  An
 * explicit num_splits always cuts the table into equal splits.  Uses the
 * current CUDA device. */
PA_API int pa_decode_num_splits(const pa_pool* pool, int S, int n_q_heads, int max_blocks_per_seq,
                         int* num_splits);

/* Device scratch bytes pa_decode needs for this shape and num_splits
 * (0: the automatic count).  Fixed splits: S * n_q_heads * splits *
 * (head_dim + 2) * 4 (each split's partial softmax states), or 0 for one
 * split, where splits is num_splits resolved against the table (at most
 * max_blocks_per_seq, and ceil(max_blocks_per_seq / ceil(max_blocks_per_seq /
 * num_splits))).  PA_SPLITS_BALANCED: ctas * (2 * G * (head_dim + 2) * 4 + 16),
 * two partial slots and one merge job per CTA, with ctas the schedule's CTAs
 * on the current device and G = n_q_heads / n_kv_heads. */
PA_API int pa_decode_workspace_bytes(const pa_pool* pool, int S, int n_q_heads, int max_blocks_per_seq,
                              int num_splits, size_t* bytes);

/* Paged decode attention, one query token per sequence, for layer `layer`.
 *   out               device [S][n_q_heads][head_dim] of out_dtype: the query
 *                     dtype (PA_FP16 for FP16 pools, PA_BF16 otherwise), or
 *                     PA_FP32 (the fp32 check mode)
 *   q                 device [S][n_q_heads][head_dim], same dtype as the
 *                     pool's inputs
 *   block_tables_dev  device int32 [S][max_blocks_per_seq]
 *   ctx_lens_dev      device int32 [S]: tokens of context of each sequence,
 *                     including the token written this step; 0 gives a zero
 *                     output row
 *   softmax_scale     multiplies q.k (usually 1/sqrt(head_dim)); any finite
 *                     value (0 weighs every visible token the same, a negative
 *                     scale takes the softmax of the negated scores), else
 *                     PA_ERR_INVALID
 *   num_splits        0 = automatic (see pa_decode_num_splits: equal splits,
 *                     or the guided layout); > 0: that many equal splits along
 *                     the pages (a second kernel merges the partial results);
 *                     PA_SPLITS_BALANCED: the balanced schedule
 *   workspace         device scratch of at least pa_decode_workspace_bytes
 *                     (may be NULL when that size is 0)
 * Query head g reads KV head g / (n_q_heads / n_kv_heads) (grouped-query
 * attention); n_q_heads / n_kv_heads must be between 1 and 8.  For each
 * sequence the result is softmax(softmax_scale * q K^T) V over its first
 * ctx_len tokens, gathered page by page through its block table ("Capítulo 8
 * ...", section 8.1).  Table entries beyond ceil(ctx_len / 16) are not read.
 * An id outside [0, num_blocks) or ctx_len > 16 * max_blocks_per_seq sets
 * PA_ERR_BOUNDS in the device error word (the output is then undefined). */
PA_API int pa_decode(pa_pool* pool, int layer, void* out, int out_dtype, const void* q,
              const int32_t* block_tables_dev, int max_blocks_per_seq, const int32_t* ctx_lens_dev,
              int S, int n_q_heads, float softmax_scale, int num_splits, void* workspace,
              size_t workspace_bytes, void* stream);

/* Size of the device scratch that pa_decode_no_alloc keeps in the library
 * itself: 8 MiB per GPU that loads the library, held until the process exits. */
#define PA_NOALLOC_SCRATCH_BYTES (8u << 20)

/* pa_decode for callers that cannot allocate device memory.  (The pages have
 * no counterpart: this is an integration entry point of this library.)
 *
 * Some callers cannot call cudaMalloc or any allocating routine: a plugin run
 * by a host framework that owns every device allocation and hands the plugin
 * only its input and output pointers, or a serving loop that must not allocate
 * once it is running, because an allocation can synchronise the device and
 * stall the other streams.  Such a caller cannot provide pa_decode's
 * workspace.  This variant takes the same arguments minus the workspace and
 * keeps the split partials in a fixed array inside the library instead, of
 * PA_NOALLOC_SCRATCH_BYTES.  It allocates nothing and frees nothing.
 *
 *  - num_splits = 0: the automatic split count, lowered until its partials
 *    fit the array (one split needs no scratch at all); the guided layout of
 *    pa_decode_num_splits when its partials fit.
 *  - num_splits = PA_SPLITS_BALANCED: at most PA_NOALLOC_SCRATCH_BYTES /
 *    (2 * G * (head_dim + 2) * 4 + 16) CTAs (more than the resident slots of
 *    a GB300 for every supported shape, so the same launch as pa_decode).
 *  - num_splits > 0: resolved against the table as for
 *    pa_decode_workspace_bytes; a resolved count whose partials,
 *    S * n_q_heads * splits * (head_dim + 2) * 4 bytes, exceed
 *    PA_NOALLOC_SCRATCH_BYTES is rejected with PA_ERR_INVALID.
 *  - The first call on a device looks up the array's device address with that
 *    device current and keeps it for the life of the process; make that first
 *    call before any stream capture, and make no call after a cudaDeviceReset
 *    of that device (the kept address would be stale).
 *  - Every call on a device shares the one array and overwrites it.  Each call
 *    writes every partial its merge reads before reading it, so nothing needs
 *    clearing between calls, but calls whose kernels overlap on the GPU (on
 *    different streams, or from different threads) race on it: serialise them.
 *  - Arguments are checked as pa_decode checks them, in the same order.
 * Results equal pa_decode's for the same schedule: bit for bit. */
PA_API int pa_decode_no_alloc(pa_pool* pool, int layer, void* out, int out_dtype, const void* q,
                              const int32_t* block_tables_dev, int max_blocks_per_seq,
                              const int32_t* ctx_lens_dev, int S, int n_q_heads,
                              float softmax_scale, int num_splits, void* stream);

/* Chunked prefill: causal attention of a chunk of new tokens per sequence over
 * its paged history ("Optimización de KV Cache ...", sections 5 and 6.3:
 * prefill split into packets, e.g. 8,192 tokens, interleaved with decode).
 * The chunk's K/V must already be in the cache (pa_reshape_and_cache).
 *   q                 device [T][n_q_heads][head_dim], the pool's query dtype;
 *                     sequence s's chunk is rows q_start[s] .. q_start[s+1]-1
 *   q_start_dev       device int32 [S+1], non-decreasing, q_start[0] = 0,
 *                     q_start[S] = T (a negative entry or a decreasing pair
 *                     sets PA_ERR_BOUNDS and that sequence is skipped; entries
 *                     above T cannot be detected and address past q and out)
 *   ctx_lens_dev      device int32 [S]: tokens of each sequence in the cache,
 *                     chunk included (>= its chunk length)
 *   out               device [T][n_q_heads][head_dim], q's dtype or PA_FP32
 *   max_chunk         an upper bound on every chunk length (sizes the grid;
 *                     rows of a longer chunk past the grid are not written
 *                     and PA_ERR_BOUNDS is set)
 *   softmax_scale     as for pa_decode
 * Query row j of a chunk of C tokens sits at position ctx - C + j and attends
 * to tokens [0, ctx - C + j] of its sequence (grouped-query heads as in
 * pa_decode).  Invalid ids or lengths set PA_ERR_BOUNDS in the device error
 * word (those rows are then not written).  The tensor-core kernel of FP8
 * pools takes its whole-tensor-memory allocation to start at column 0; a CTA
 * that finds otherwise sets PA_ERR_UNSUPPORTED and writes nothing.  No
 * scratch memory is needed. */
PA_API int pa_prefill(pa_pool* pool, int layer, void* out, int out_dtype, const void* q,
                      const int32_t* q_start_dev, const int32_t* block_tables_dev,
                      int max_blocks_per_seq, const int32_t* ctx_lens_dev, int S, int n_q_heads,
                      int max_chunk, float softmax_scale, void* stream);

/* For tests of the timeout path only: sets, for the current device, how long
 * the kernels' pipeline waits (a stage's data, a free stage, a hand-off
 * between warp roles) spin before they give up, record PA_ERR_TIMEOUT and
 * unwind.  0 restores the default of 2 s.  The waits that drain copies
 * already in flight before a CTA exits always keep 2 s.  Blocking: it copies
 * the value into each kernel module's device variable; it holds for every
 * later launch in the process until it is set again.  (The pages have no
 * counterpart: the bound itself is what keeps a stalled pipeline from hanging
 * the GPU.) */
PA_API int pa_set_pipeline_wait_limit_ns(uint64_t ns);

/* Synchronises `stream`, then reads and clears the current device's error word.
 * *code = PA_OK or the first PA_ERR_* a kernel recorded since the last read.
 * The word is shared by every pool on the device. */
PA_API int pa_get_device_error(pa_pool* pool, int* code, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_PA_H */
