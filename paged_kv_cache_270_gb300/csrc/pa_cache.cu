// pa_cache.cu -- writing into the paged KV pool: scatter of new tokens into
// their slots (with on-the-fly FP8 E4M3 quantisation) and whole-block copies
// for copy-on-write.  Also owns the per-device error word.
//
// New tokens fill pages on demand through the slot mapping ("Optimización de
// KV Cache con PagedAttention y Cuantización FP8 para Contextos Largos
// (128K)", section 3: pages are assigned and linked dynamically); an FP8 cache
// converts each 16-bit value to 8 bits as it is written (same page, section
// 4) with a static per-tensor scale (section 8, static calibration).  Block
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
// copy_blocks: blockIdx.y = pair; the K and V bytes of the whole block (all
// kv heads of one layer) are copied as 16-byte vectors.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const int32_t* __restrict__ pairs,
                                                          int num_blocks, long long block_vecs,
                                                          uint4* kpool, uint4* vpool,
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
}

// ---------------------------------------------------------------------------
// swap: blockIdx.x = block i of the list, blockIdx.y = layer * 2 + (0: K, 1: V).
// One region = the block's tiles of every kv head in one layer, contiguous in
// the pool and in the host buffer.  `to_host` selects the direction.
__global__ void __launch_bounds__(256) swap_kernel(const int32_t* __restrict__ ids, int num_blocks,
                                                   uint4* kpool, uint4* vpool,
                                                   long long layer_vecs, long long region_vecs,
                                                   uint4* host, int to_host, unsigned int* err) {
  const int i = blockIdx.x;
  const int layer = blockIdx.y >> 1, which = blockIdx.y & 1;
  const int b = ids[i];
  if (b < 0 || b >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) record_error(err, PA_ERR_BOUNDS);
    return;
  }
  uint4* pool = (which ? vpool : kpool) + layer * layer_vecs + (long long)b * region_vecs;
  uint4* h = host + ((long long)i * gridDim.y + blockIdx.y) * region_vecs;
  if (to_host) {
    for (long long v = threadIdx.x; v < region_vecs; v += blockDim.x) h[v] = pool[v];
  } else {
    for (long long v = threadIdx.x; v < region_vecs; v += blockDim.x) pool[v] = h[v];
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
  swap_kernel<<<dim3(n, pool->desc.n_layers * 2), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      ids_dev, pool->desc.num_blocks, reinterpret_cast<uint4*>(pool->k),
      reinterpret_cast<uint4*>(pool->v), layer_vecs, region_vecs, static_cast<uint4*>(dev_view),
      to_host, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "swap launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

extern "C" {

int pa_reshape_and_cache(pa_pool* pool, int layer, const void* k, const void* v,
                         const int64_t* slot_mapping_dev, int T, void* stream) {
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
  if (d.kv_dtype == PA_FP8_E4M3) {
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
  copy_blocks_kernel<<<dim3(gx, n_pairs), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      pairs_dev, pool->desc.num_blocks, block_vecs, reinterpret_cast<uint4*>(kp),
      reinterpret_cast<uint4*>(vp), err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "copy_blocks launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

int pa_swap_block_bytes(const pa_pool* pool, size_t* bytes) {
  if (!pool || !bytes) return fail(PA_ERR_INVALID, "null argument");
  *bytes = 2ull * pool->desc.n_layers * pool->desc.n_kv_heads * pool->tile_bytes;
  return PA_OK;
}

int pa_swap_out(pa_pool* pool, int n, const int32_t* ids_dev, void* host_buf, void* stream) {
  return swap_common(pool, n, ids_dev, host_buf, 1, stream);
}

int pa_swap_in(pa_pool* pool, int n, const int32_t* ids_dev, const void* host_buf, void* stream) {
  return swap_common(pool, n, ids_dev, host_buf, 0, stream);
}

int pa_get_device_error(pa_pool* pool, int* code, void* stream) {
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
