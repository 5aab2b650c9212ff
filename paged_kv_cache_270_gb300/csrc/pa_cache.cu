// pa_cache.cu -- writing into the paged KV pool: scatter of new tokens into
// their slots (with on-the-fly FP8 E4M3 quantisation, static or per block),
// whole-block copies for copy-on-write, and block swaps to host memory.  Also
// owns the per-device error word.
//
// New tokens fill pages on demand through the slot mapping ("Optimización de
// KV Cache con PagedAttention y Cuantización FP8 para Contextos Largos
// (128K)", section 3: pages are assigned and linked dynamically); an FP8 cache
// converts each 16-bit value to 8 bits as it is written (same page, section
// 4) with a static per-tensor scale (section 8, static calibration) or with a
// scale per block taken from the block's MaxAbs (section 8, dynamic scaling).  Block
// copies are the device half of copy-on-write for shared prefixes and
// branches ("PagedAttention y Gestión de KV-Cache", sections 3.01, 3.02).
#include <cuda_runtime.h>

#include <mutex>

#include "pa_device.cuh"

namespace pa {

__device__ unsigned int g_device_error;  // one per device; 0 = no error

unsigned int* device_error_word() {
  static std::mutex mu;
  static unsigned int* cached[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 128) {
    fail(PA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) {
      fail(PA_ERR_CUDA, "cudaGetSymbolAddress(error word): %s", cudaGetErrorString(e));
      return nullptr;
    }
    cached[dev] = static_cast<unsigned int*>(p);
  }
  return cached[dev];
}

// ---------------------------------------------------------------------------
// reshape_and_cache: one thread per 8 consecutive elements of one (token,
// kv head) row.  Inputs are read as 16-byte vectors; a 16-bit cache receives
// them unchanged, an FP8 cache receives E4M3(fl32(x / scale)), rounded to
// nearest-even and saturated to +-448.
template <bool FP8>
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, const int64_t* __restrict__ slots,
    long long n_vec, int vec_per_token, int vec_per_row, int head_dim, long long num_slots,
    uint8_t* __restrict__ kpool, uint8_t* __restrict__ vpool, float k_scale, float v_scale,
    unsigned int* err) {
  // A decode launched behind this kernel (programmatic stream serialization)
  // may be scheduled now: it waits for this grid's completion and its writes
  // before its first global access, so only its launch and CTA placement
  // overlap this kernel.
  grid_dependents_launch();
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_vec) return;
  const long long t = i / vec_per_token;
  const int r = (int)(i - t * vec_per_token);
  const int h = r / vec_per_row;
  const int c = r - h * vec_per_row;
  const int64_t slot = slots[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    record_error(err, PA_ERR_BOUNDS);
    return;
  }
  const int n_kv_heads = vec_per_token / vec_per_row;
  const long long blk = slot >> 4;
  const int off = (int)(slot & 15);
  // element index of (blk, h, off, 8c) in [num_blocks][n_kv_heads][16][head_dim]
  const long long e = ((blk * n_kv_heads + h) * 16 + off) * (long long)head_dim + 8 * c;
  const uint4 kx = k[i];
  const uint4 vx = v[i];
  if constexpr (!FP8) {
    *reinterpret_cast<uint4*>(kpool + 2 * e) = kx;
    *reinterpret_cast<uint4*>(vpool + 2 * e) = vx;
  } else {
    const uint32_t kw[4] = {kx.x, kx.y, kx.z, kx.w};
    const uint32_t vw[4] = {vx.x, vx.y, vx.z, vx.w};
    uint32_t ko[2], vo[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t kq[2], vq[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint32_t kwrd = kw[2 * j + h2], vwrd = vw[2 * j + h2];
        float2 kf = make_float2(__fdiv_rn(bf16_bits_to_float(kwrd & 0xFFFFu), k_scale),
                                __fdiv_rn(bf16_bits_to_float(kwrd >> 16), k_scale));
        float2 vf = make_float2(__fdiv_rn(bf16_bits_to_float(vwrd & 0xFFFFu), v_scale),
                                __fdiv_rn(bf16_bits_to_float(vwrd >> 16), v_scale));
        kq[h2] = __nv_cvt_float2_to_fp8x2(kf, __NV_SATFINITE, __NV_E4M3);
        vq[h2] = __nv_cvt_float2_to_fp8x2(vf, __NV_SATFINITE, __NV_E4M3);
      }
      ko[j] = kq[0] | (kq[1] << 16);
      vo[j] = vq[0] | (vq[1] << 16);
    }
    *reinterpret_cast<uint2*>(kpool + e) = make_uint2(ko[0], ko[1]);
    *reinterpret_cast<uint2*>(vpool + e) = make_uint2(vo[0], vo[1]);
  }
}

// ---------------------------------------------------------------------------
// reshape_and_cache of a block-scaled FP8 pool (dynamic scaling: the MaxAbs of
// each block taken as it is written).  One CTA per (token, kv head); only the
// CTA of the first token of a run -- the tokens after it in the slot mapping
// whose slots follow it within its block -- does the work, for the whole run:
//   m = max |x| of the run, s_run = fl32(m / 448);
//   run at offset 0: s = s_run; else s = max(s_old, s_run), and if s grew the
//   earlier rows' codes c become E4M3(fl32(fl32(decode(c) * s_old) / s));
//   the run's values become E4M3(fl32(x / s)) (0 when s = 0); s is stored.

// largest |x| of 8 bfloat16 values: without the sign bit, bf16 magnitudes
// order like their bit patterns
__device__ __forceinline__ uint32_t absmax_bits8(uint4 x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  return m;
}

// E4M3 codes of 8 bfloat16 values x / s (code 0 when s = 0)
__device__ __forceinline__ uint2 quantize8(uint4 x, float s) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = make_float2(0.f, 0.f);
    if (s > 0.f)
      f = make_float2(__fdiv_rn(bf16_bits_to_float(w[i] & 0xFFFFu), s),
                      __fdiv_rn(bf16_bits_to_float(w[i] >> 16), s));
    q[i] = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
  }
  return make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
}

// Re-encodes `words` 8-byte groups of codes from scale s_old to s_new.
__device__ __forceinline__ void requantize(uint8_t* tile, int words, float s_old, float s_new) {
  for (int i = threadIdx.x; i < words; i += blockDim.x) {
    uint2* p = reinterpret_cast<uint2*>(tile) + i;
    const uint2 c = *p;
    const uint32_t cw[2] = {c.x, c.y};
    uint32_t o[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t q[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
            static_cast<__nv_fp8x2_storage_t>((cw[j] >> (16 * hh)) & 0xFFFFu), __NV_E4M3);
        const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        const float2 f = make_float2(__fdiv_rn(__fmul_rn(y.x, s_old), s_new),
                                     __fdiv_rn(__fmul_rn(y.y, s_old), s_new));
        q[hh] = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      }
      o[j] = q[0] | (q[1] << 16);
    }
    *p = make_uint2(o[0], o[1]);
  }
}

template <int D>
__global__ void __launch_bounds__(128) reshape_block_scaled_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
    const int64_t* __restrict__ slots, int T, int n_kv_heads, long long num_slots,
    uint8_t* __restrict__ kpool, uint8_t* __restrict__ vpool, float* __restrict__ ksc,
    float* __restrict__ vsc, unsigned int* err) {
  __shared__ uint32_t red[2][4];
  grid_dependents_launch();  // (as in reshape_and_cache_kernel)
  const int t = blockIdx.x, h = blockIdx.y;
  const int64_t slot = slots[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0 && h == 0) record_error(err, PA_ERR_BOUNDS);
    return;
  }
  const int off0 = (int)(slot & 15);
  if (t > 0 && off0 != 0 && slots[t - 1] == slot - 1) return;  // not the first token of its run
  int n = 1;
  while (n < 16 - off0 && t + n < T && slots[t + n] == slot + n) ++n;
  const long long blk = slot >> 4;
  const size_t sidx = (size_t)blk * n_kv_heads + h;
  // the stored scales are read before the barrier below, written after it
  const float sk_old = off0 > 0 ? ksc[sidx] : 0.f;
  const float sv_old = off0 > 0 ? vsc[sidx] : 0.f;

  constexpr int VPR = D / 8;  // 16-byte vectors per row
  const int nvec = n * VPR;
  uint32_t mk = 0, mv = 0;
  for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
    const int r = i / VPR, c = i - r * VPR;
    const size_t src = ((size_t)(t + r) * n_kv_heads + h) * D + 8 * c;
    mk = max(mk, absmax_bits8(*reinterpret_cast<const uint4*>(k + src)));
    mv = max(mv, absmax_bits8(*reinterpret_cast<const uint4*>(v + src)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, o));
    mv = max(mv, __shfl_xor_sync(0xffffffffu, mv, o));
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = mk;
    red[1][threadIdx.x >> 5] = mv;
  }
  __syncthreads();
  mk = max(max(red[0][0], red[0][1]), max(red[0][2], red[0][3]));
  mv = max(max(red[1][0], red[1][1]), max(red[1][2], red[1][3]));
  const float sk_run = __fdiv_rn(bf16_bits_to_float(mk), 448.f);
  const float sv_run = __fdiv_rn(bf16_bits_to_float(mv), 448.f);
  const bool grow_k = off0 == 0 || sk_run > sk_old, grow_v = off0 == 0 || sv_run > sv_old;
  const float sk = grow_k ? sk_run : sk_old, sv = grow_v ? sv_run : sv_old;

  const size_t tile = sidx * 16 * D;  // byte offset of the (block, head) tile
  if (off0 > 0 && grow_k) requantize(kpool + tile, off0 * D / 8, sk_old, sk);
  if (off0 > 0 && grow_v) requantize(vpool + tile, off0 * D / 8, sv_old, sv);
  for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
    const int r = i / VPR, c = i - r * VPR;
    const size_t src = ((size_t)(t + r) * n_kv_heads + h) * D + 8 * c;
    const size_t dst = tile + (size_t)(off0 + r) * D + 8 * c;
    *reinterpret_cast<uint2*>(kpool + dst) = quantize8(*reinterpret_cast<const uint4*>(k + src), sk);
    *reinterpret_cast<uint2*>(vpool + dst) = quantize8(*reinterpret_cast<const uint4*>(v + src), sv);
  }
  if (threadIdx.x == 0) {
    ksc[sidx] = sk;
    vsc[sidx] = sv;
  }
}

// ---------------------------------------------------------------------------
// copy_blocks: blockIdx.y = pair; the K and V bytes of the whole block (all
// kv heads of one layer) are copied as 16-byte vectors, and for block-scaled
// pools (ksc != nullptr) the block's n_kv_heads K and V scales.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const int32_t* __restrict__ pairs,
                                                          int num_blocks, long long block_vecs,
                                                          uint4* kpool, uint4* vpool, float* ksc,
                                                          float* vsc, int n_kv_heads,
                                                          unsigned int* err) {
  const int p = blockIdx.y;
  const int src = pairs[2 * p], dst = pairs[2 * p + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_error(err, PA_ERR_BOUNDS);
    return;
  }
  const uint4* ks = kpool + (long long)src * block_vecs;
  const uint4* vs = vpool + (long long)src * block_vecs;
  uint4* kd = kpool + (long long)dst * block_vecs;
  uint4* vd = vpool + (long long)dst * block_vecs;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < block_vecs;
       i += (long long)gridDim.x * blockDim.x) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
  if (ksc && blockIdx.x == 0) {
    for (int i = threadIdx.x; i < n_kv_heads; i += blockDim.x) {
      ksc[(size_t)dst * n_kv_heads + i] = ksc[(size_t)src * n_kv_heads + i];
      vsc[(size_t)dst * n_kv_heads + i] = vsc[(size_t)src * n_kv_heads + i];
    }
  }
}

// ---------------------------------------------------------------------------
// swap: blockIdx.x = block i of the list, blockIdx.y = layer * 2 + (0: K, 1: V).
// One region = the block's tiles of every kv head in one layer, contiguous in
// the pool and in the host buffer; a block's record is its regions, then for
// block-scaled pools (ksc != nullptr) its scales [layer][K|V][n_kv_heads] and
// zero padding to record_vecs.  `to_host` selects the direction.
__global__ void __launch_bounds__(256) swap_kernel(const int32_t* __restrict__ ids, int num_blocks,
                                                   uint4* kpool, uint4* vpool,
                                                   long long layer_vecs, long long region_vecs,
                                                   long long record_vecs, float* ksc, float* vsc,
                                                   int n_kv_heads, uint4* host, int to_host,
                                                   unsigned int* err) {
  const int i = blockIdx.x;
  const int layer = blockIdx.y >> 1, which = blockIdx.y & 1;
  const int b = ids[i];
  if (b < 0 || b >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) record_error(err, PA_ERR_BOUNDS);
    return;
  }
  uint4* pool = (which ? vpool : kpool) + layer * layer_vecs + (long long)b * region_vecs;
  uint4* rec = host + (long long)i * record_vecs;
  uint4* h = rec + (long long)blockIdx.y * region_vecs;
  if (to_host) {
    for (long long v = threadIdx.x; v < region_vecs; v += blockDim.x) h[v] = pool[v];
  } else {
    for (long long v = threadIdx.x; v < region_vecs; v += blockDim.x) pool[v] = h[v];
  }
  if (ksc) {
    float* hs = reinterpret_cast<float*>(rec + (long long)gridDim.y * region_vecs);
    float* ps = (which ? vsc : ksc) + ((size_t)layer * num_blocks + b) * n_kv_heads;
    float* hh = hs + (size_t)blockIdx.y * n_kv_heads;
    for (int j = threadIdx.x; j < n_kv_heads; j += blockDim.x) {
      if (to_host) hh[j] = ps[j];
      else ps[j] = hh[j];
    }
    if (to_host && blockIdx.y == 0) {  // zero the padding after the last scale
      const long long used = (long long)gridDim.y * n_kv_heads;
      const long long words = (record_vecs - (long long)gridDim.y * region_vecs) * 4;
      for (long long j = used + threadIdx.x; j < words; j += blockDim.x) hs[j] = 0.f;
    }
  }
}

}  // namespace pa

using namespace pa;

static int swap_common(pa_pool* pool, int n, const int32_t* ids_dev, const void* host_buf,
                       int to_host, void* stream) {
  if (!pool) return fail(PA_ERR_INVALID, "null pool");
  if (n < 0) return fail(PA_ERR_INVALID, "n must be >= 0");
  if (n == 0) return PA_OK;
  if (!ids_dev || !host_buf) return fail(PA_ERR_INVALID, "null argument");
  if (n > 0x7FFFFFFF / 2 || pool->desc.n_layers * 2 > 65535)
    return fail(PA_ERR_UNSUPPORTED, "too many blocks or layers for one swap call");
  // Only page-locked host memory is accepted: on systems where the GPU can also
  // reach pageable memory, a pageable buffer would otherwise be written directly.
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, host_buf);
  if (e != cudaSuccess || attr.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    return fail(PA_ERR_INVALID, "swap buffer is not page-locked host memory");
  }
  void* dev_view = attr.devicePointer;
  if (!dev_view) {
    e = cudaHostGetDevicePointer(&dev_view, const_cast<void*>(host_buf), 0);
    if (e != cudaSuccess || !dev_view) {
      cudaGetLastError();
      return fail(PA_ERR_INVALID, "swap buffer is not device-accessible");
    }
  }
  if ((uintptr_t)dev_view & 15u) return fail(PA_ERR_INVALID, "swap buffer must be 16-byte aligned");
  unsigned int* err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  const long long region_vecs = (long long)pool->desc.n_kv_heads * pool->tile_bytes / 16;
  const long long layer_vecs = (long long)pool->layer_bytes / 16;
  size_t record = 0;
  pa_swap_block_bytes(pool, &record);
  float* ksc = pool->block_scaled ? layer_scales(pool, pool->k, 0) : nullptr;
  float* vsc = pool->block_scaled ? layer_scales(pool, pool->v, 0) : nullptr;
  swap_kernel<<<dim3(n, pool->desc.n_layers * 2), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      ids_dev, pool->desc.num_blocks, reinterpret_cast<uint4*>(pool->k),
      reinterpret_cast<uint4*>(pool->v), layer_vecs, region_vecs, (long long)(record / 16), ksc,
      vsc, pool->desc.n_kv_heads, static_cast<uint4*>(dev_view), to_host, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "swap launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

extern "C" {

int pa_reshape_and_cache(pa_pool* pool, int layer, const void* k, const void* v,
                         const int64_t* slot_mapping_dev, int T, void* stream) {
  pa::TraceRange trace_("pa_reshape_and_cache");
  int st = check_pool_layer(pool, layer);
  if (st) return st;
  if (T < 0) return fail(PA_ERR_INVALID, "T must be >= 0");
  if (T == 0) return PA_OK;
  if (!k || !v || !slot_mapping_dev) return fail(PA_ERR_INVALID, "null input");
  if (((uintptr_t)k | (uintptr_t)v) & 15u) return fail(PA_ERR_INVALID, "k and v must be 16-byte aligned");
  unsigned int* err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  const pa_pool_desc& d = pool->desc;
  const int vec_per_row = d.head_dim / 8;
  const int vec_per_token = d.n_kv_heads * vec_per_row;
  const long long n_vec = (long long)T * vec_per_token;
  const long long blocks = (n_vec + 255) / 256;
  uint8_t* kp = pool->k + (size_t)layer * pool->layer_bytes;
  uint8_t* vp = pool->v + (size_t)layer * pool->layer_bytes;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pool->block_scaled) {
    const dim3 grid((unsigned)T, (unsigned)d.n_kv_heads);
    if (d.n_kv_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "at most 65535 kv heads");
    auto kern = d.head_dim == 64 ? reshape_block_scaled_kernel<64> : reshape_block_scaled_kernel<128>;
    kern<<<grid, 128, 0, s>>>(static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v),
                              slot_mapping_dev, T, d.n_kv_heads, (long long)d.num_blocks * 16, kp,
                              vp, layer_scales(pool, pool->k, layer),
                              layer_scales(pool, pool->v, layer), err);
  } else if (d.kv_dtype == PA_FP8_E4M3) {
    reshape_and_cache_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping_dev, n_vec,
        vec_per_token, vec_per_row, d.head_dim, (long long)d.num_blocks * 16, kp, vp, d.k_scale,
        d.v_scale, err);
  } else {
    reshape_and_cache_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping_dev, n_vec,
        vec_per_token, vec_per_row, d.head_dim, (long long)d.num_blocks * 16, kp, vp, 1.f, 1.f,
        err);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "reshape_and_cache launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

int pa_copy_blocks(pa_pool* pool, int layer, const int32_t* pairs_dev, int n_pairs, void* stream) {
  pa::TraceRange trace_("pa_copy_blocks");
  int st = check_pool_layer(pool, layer);
  if (st) return st;
  if (n_pairs < 0) return fail(PA_ERR_INVALID, "n_pairs must be >= 0");
  if (n_pairs == 0) return PA_OK;
  if (!pairs_dev) return fail(PA_ERR_INVALID, "null pairs");
  if (n_pairs > 65535) return fail(PA_ERR_UNSUPPORTED, "at most 65535 pairs per call");
  unsigned int* err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  const long long block_vecs = (long long)pool->desc.n_kv_heads * pool->tile_bytes / 16;
  const int gx = (int)((block_vecs + 255) / 256 < 8 ? (block_vecs + 255) / 256 : 8);
  uint8_t* kp = pool->k + (size_t)layer * pool->layer_bytes;
  uint8_t* vp = pool->v + (size_t)layer * pool->layer_bytes;
  float* ksc = pool->block_scaled ? layer_scales(pool, pool->k, layer) : nullptr;
  float* vsc = pool->block_scaled ? layer_scales(pool, pool->v, layer) : nullptr;
  copy_blocks_kernel<<<dim3(gx, n_pairs), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      pairs_dev, pool->desc.num_blocks, block_vecs, reinterpret_cast<uint4*>(kp),
      reinterpret_cast<uint4*>(vp), ksc, vsc, pool->desc.n_kv_heads, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "copy_blocks launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

int pa_swap_block_bytes(const pa_pool* pool, size_t* bytes) {
  if (!pool || !bytes) return fail(PA_ERR_INVALID, "null argument");
  *bytes = 2ull * pool->desc.n_layers * pool->desc.n_kv_heads * pool->tile_bytes;
  if (pool->block_scaled)
    *bytes += (2ull * pool->desc.n_layers * pool->desc.n_kv_heads * sizeof(float) + 15) / 16 * 16;
  return PA_OK;
}

int pa_swap_out(pa_pool* pool, int n, const int32_t* ids_dev, void* host_buf, void* stream) {
  pa::TraceRange trace_("pa_swap_out");
  return swap_common(pool, n, ids_dev, host_buf, 1, stream);
}

int pa_swap_in(pa_pool* pool, int n, const int32_t* ids_dev, const void* host_buf, void* stream) {
  pa::TraceRange trace_("pa_swap_in");
  return swap_common(pool, n, ids_dev, host_buf, 0, stream);
}

int pa_get_device_error(pa_pool* pool, int* code, void* stream) {
  pa::TraceRange trace_("pa_get_device_error");
  (void)pool;
  if (!code) return fail(PA_ERR_INVALID, "null output");
  *code = PA_OK;
  unsigned int* err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, err, sizeof h, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof h, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(e));
  *code = (int)h;
  return PA_OK;
}

}  // extern "C"
