// pa_device.cuh -- device-side building blocks for the sm_103a kernels:
// mbarrier-tracked bulk (TMA) copies, bounded waits, warp-level tensor-core
// MMA, fragment transposes and FP8 conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pa_internal.h"

namespace pa {

// ---------------------------------------------------------------- errors
// First error wins; later ones are dropped (the host reads one code).
__device__ __forceinline__ void record_error(unsigned int* err, unsigned int code) {
  if (err) atomicCAS(err, 0u, code);
}

// ---------------------------------------------------------------- timing
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every spin-wait in the library gives up after this long and reports
// PA_ERR_TIMEOUT instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// The limit of the pipeline waits (a stage's data, a free stage, a role's
// hand-off).  Tests of the timeout path lower it through
// pa_set_pipeline_wait_limit_ns; the waits that drain copies already in flight
// before a CTA exits keep kWaitLimitNs.  One copy per translation unit.
static __device__ unsigned long long g_pipe_wait_ns = kWaitLimitNs;

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete; false after
// `limit` ns (the caller then records PA_ERR_TIMEOUT and unwinds).  The drain
// waits use the default; the pipeline waits pass pipe_wait_limit().
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit) return false;
  }
  return true;
}

__device__ __forceinline__ uint64_t pipe_wait_limit() { return g_pipe_wait_ns; }

// Host side: sets this translation unit's pipeline wait limit (0: the default).
static inline cudaError_t set_pipe_wait_limit_here(unsigned long long ns) {
  const unsigned long long v = ns ? ns : kWaitLimitNs;
  return cudaMemcpyToSymbol(g_pipe_wait_ns, &v, sizeof(v));
}

// ---------------------------------------------------------------- bulk copy
// One-dimensional bulk copy global -> shared by the TMA unit, completing
// `bytes` of transaction count on `bar`.  Addresses 16-B aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Tiled tensor copies global -> shared through a tensor map (TMA), completing
// on `bar`.  The map lives in kernel-parameter space (__grid_constant__).
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int c0, int c1,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int c0, int c1, int c2,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy (bulk copy) accesses to it, once the threads meet at a barrier.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// Byte offset inside a 1024-byte-aligned tile written by a TMA copy with
// 128-byte swizzling: the 16-byte chunk index (bits 4-6) is XORed with the
// 128-byte line index (bits 7-9).
__device__ __forceinline__ uint32_t swizzle128(uint32_t off) { return off ^ ((off >> 3) & 0x70u); }

// 2^x on the SFU (max relative error ~2^-22); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// L2 policy for data streamed exactly once (the KV tiles of a decode pass).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- shared loads
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

__device__ __forceinline__ uint2 lds64(const void* p) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_addr(p)));
  return v;
}

// ---------------------------------------------------------------- dependent launch
// A kernel launched with programmatic stream serialization may start while the
// kernel before it in the stream is still running.  It must wait here, before
// touching global memory that kernel may write or read; the wait returns once
// that grid has completed and its writes are visible (at once for an ordinary
// launch).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream, if launched that way, be scheduled once
// every CTA of this grid has called this or exited.
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- MMA
// D(16x8, fp32) += A(16x16, row) * B(16x8, col), warp-wide.
// Fragment ownership (g = lane / 4, t = lane % 4):
//   a[0] = A[g][2t..2t+1]     a[1] = A[g+8][2t..2t+1]
//   a[2] = A[g][2t+8..2t+9]   a[3] = A[g+8][2t+8..2t+9]
//   b[0] = B[2t..2t+1][g]     b[1] = B[2t+8..2t+9][g]
//   c[0..1] = D[g][2t..2t+1]  c[2..3] = D[g+8][2t..2t+1]
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (BF16) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Two 16 x 16 byte matrices from shared memory, transposed: lanes 0-15 give the
// addresses of the first matrix's 16 rows (16 bytes each), lanes 16-31 those of
// the second.  Lane 4g + t receives rows 4t .. 4t+3 of column g (r0) and of
// column g + 8 (r1) of the first matrix, low byte = row 4t, and the same of
// the second in (r2, r3).
__device__ __forceinline__ void ldsm_x2_trans_b8(const void* row, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                 uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_addr(row)));
}

// Four 8 x 8 matrices of 16-bit elements from shared memory, transposed: lanes
// 8m .. 8m+7 give the addresses of matrix m's 8 rows (16 bytes each).  Lane
// 4g + t receives rows 2t and 2t+1 of column g of matrix m in rm (low half =
// row 2t).
__device__ __forceinline__ void ldsm_x4_trans_b16(const void* row, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_addr(row)));
}

// Transpose of an 8x8 matrix of 16-bit elements held one row-pair per lane
// (lane 4r + c holds row r, columns 2c and 2c+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// ---------------------------------------------------------------- conversions
// E4M3 codes -> binary16, exact (low byte / low half first).  The conversion
// instruction takes a 16-bit register; the 32-bit word is split into its two
// halves as registers, which costs no instruction, where a shift or mask of
// the word to reach its upper pair would (measured on the decode kernel: the
// split form is 10-14% faster there).
// Two codes in the low half of the word -> one binary16 pair.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t}" : "=r"(r) : "r"(two_codes));
  return r;
}
// Four codes -> the binary16 pairs of codes (0, 1) in lo and (2, 3) in hi.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi) : "r"(four));
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t x) {
  if constexpr (BF16) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&x);
    return __bfloat1622float2(v);
  } else {
    __half2 v = *reinterpret_cast<__half2*>(&x);
    return __half22float2(v);
  }
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

}  // namespace pa
