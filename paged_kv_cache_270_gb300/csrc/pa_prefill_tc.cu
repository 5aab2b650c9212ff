// pa_prefill_tc.cu -- chunked prefill over a paged KV cache on the
// fifth-generation tensor cores (tcgen05 MMA, accumulators in tensor memory).
//
// Same operation as pa_prefill.cu: a chunk of new tokens per sequence, already
// in the cache, attends causally to the sequence's pages ("Optimización de KV
// Cache con PagedAttention y Cuantización FP8 para Contextos Largos (128K)",
// sections 5 and 6.3: prefill in packets interleaved with decode; "Capítulo 8
// -- Gestión de caché KV de nueva generación", section 8.1: pages gathered
// through the block table).  This kernel takes the shapes where a CTA's rows
// fill a 128-row MMA: head_dim 128 and G = 1, 2, 4 or 8 query heads per KV
// head (a tile of 128 / G query tokens x G heads), FP8 E4M3 pages with a
// per-tensor or per-tile scale, or bfloat16 / binary16 pages.
//
// Design (the pages give none):
//  * grid = (query tile, kv head, sequence), longest tiles first; one CTA per
//    SM (131 KB of shared memory for FP8 pools, 197 KB for 16-bit pools; 448 of
//    the 512 TMEM columns: S twice, O, Q).
//  * warp 0 streams the K and V pages of 128-key blocks (8 pages) with TMA into
//    a two-block ring; the K pages land 128-byte swizzled, back to back, which
//    is exactly the K-major operand layout of the MMA, so S = Q K^T reads them
//    in place (kind::f8f6f4, M = N = 128, fp32 accumulate in TMEM).
//  * Q is FP8 too: each bf16 query row is scaled by a power of two and split
//    into two E4M3 terms, hi = E4M3(x) and lo = E4M3(x - hi); their sum
//    carries the row's 8 significant bits, so S = hi K^T + lo K^T (two MMA
//    passes into one accumulator) is exact up to fp32 accumulation order.
//  * four warps convert each V block to binary16 (exact), laid out 128-byte
//    swizzled with the head dim contiguous, which the MMA reads as its B
//    operand in MN-major form: O += P V is kind::f16 with P in binary16 (plus
//    a second pass with P's low part in the fp32-output mode).
//  * eight warps run the online softmax, two threads per row (each takes half
//    of every key block and of the row's O): S comes out of TMEM, the max moves
//    only when it grows by more than 2^8 (so P <= 2^8), and then the threads
//    rescale their halves of the O row in TMEM before the next P V.
//  * 16-bit pools take the same pipeline without the conversion: a page
//    arrives as two 64-dim halves (two TMA boxes of 128-byte rows), which is
//    at once the K-major layout of K and the MN-major layout of V, so both
//    MMAs read the ring in place (Q in TMEM unsplit; P in the pool's type, with
//    its low part whenever P in bfloat16 would be too coarse).  The ring has
//    three slots, as a V slot stays busy until its P V is done; the converter
//    warps only zero the last block's V rows past the tile.
//  * warp 1 allocates TMEM and one lane issues every MMA; completion is
//    signalled through mbarriers (tcgen05.commit).  Every wait is bounded: a
//    timeout records PA_ERR_TIMEOUT, raises a CTA-wide abort flag that ends
//    every role's loop, and the CTA drains its MMAs and copies before it frees
//    TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "pa_device.cuh"

namespace pa {
namespace {

constexpr int kD = 128;         // head dim
constexpr int kRows = 128;      // MMA rows of a tile: query tokens x the G heads of a kv head
constexpr int kThreads = 448;   // 14 warps: producer, MMA, 4 converters, 8 softmax
constexpr unsigned kAll = 0xffffffffu;
constexpr uint32_t kTmemCols = 512;
// TMEM columns (one lane per row): S(j) in buffer j % 2 at 0 / 128, overwritten
// by P(j) in 16 bits: keys 32c .. 32c+31 in columns 32c .. 32c+15 of the buffer
// (P's low part, where used, in 32c+16 .. 32c+31); O at 256; Q at 384 .. 447
// (FP8 pools: its two E4M3 terms at 384 and 416; 16-bit pools: Q itself).
constexpr uint32_t kOCol = 256;
constexpr uint32_t kQHiCol = 384;
constexpr uint32_t kQLoCol = 416;

// Cache types this kernel takes
enum Kind { K_E4M3 = 0, K_E4M3B = 1, K_BF16 = 2, K_F16 = 3 };

struct Ctrl {
  uint64_t kv_full[3], kv_empty[3], s_full[2], vt_full[2], vt_empty[2];
  // p_full is two barriers (by block parity) although one P is consumed at a
  // time: the softmax may store P(j) and P(j + 1) before the MMA thread wakes
  // for P(j) (both S were issued before that wait), and one barrier would then
  // have completed two phases, which a parity wait cannot tell from none (the
  // thread waited out its limit on one such call).  P(j + 2) needs S(j + 2),
  // issued only after P V(j), so a barrier per parity is never two phases
  // ahead of its waiter.  (Every other barrier here has that property by
  // construction.)
  uint64_t sc_full[2], sc_empty[2], p_full[2], q_ready, drain, xchg;
  uint64_t tail_ready, tail_done;  // 16-bit pools: the last block's V rows past the tile are zeroed
  float2 sc[2][8];  // block-scaled pools: (K scale, V scale) of each page of a ring block
  float xbuf[2][128][2];  // the two half-row threads' partials (Q amax, block max, row sum)
  uint32_t tmem;
  int abort;
};

// Shared memory, from a 1024-byte aligned base.  A ring slot holds one
// 128-key block (8 pages) of K and of V as the TMA wrote them, 128-byte
// swizzled.  FP8: K and V slots of 16 KiB ([8 pages][16 keys][128 B]), two
// slots, plus two binary16 V blocks converted for the MMA ([2 dim blocks][128
// keys][128 B]).  16-bit pools: each page arrives as two 64-dim halves, so a
// slot is [2 dim halves][128 keys][128 B] (32 KiB) -- the K-major layout for
// K and the MN-major layout for V, both read in place; three slots, as a V
// slot is held until its P V is done.
template <int KIND>
struct Lay {
  static constexpr bool kF8 = KIND == K_E4M3 || KIND == K_E4M3B;
  static constexpr bool kBlk = KIND == K_E4M3B;
  static constexpr bool kBf = KIND == K_BF16;
  static constexpr int kRing = kF8 ? 2 : 3;  // (a third FP8 slot measured +0.3%: not worth 32 KiB)
  static constexpr int kSlot = kF8 ? 16384 : 32768;
  static constexpr int kKRing = 0;
  static constexpr int kVRing = kRing * kSlot;
  static constexpr int kVT = kVRing + kRing * kSlot;
  static constexpr int kData = kF8 ? kVT + 65536 : kVT;
  static constexpr int kSmem = 1024 + kData + (int)sizeof(Ctrl);
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct TcArgs {
  const uint16_t* q;
  void* out;
  const int32_t* q_start;
  const int32_t* ctx;
  const int32_t* tables;
  const float* ksc;  // block-scaled pools: this layer's scales [num_blocks][Hkv]
  const float* vsc;
  int max_blocks, Hq, Hkv, num_blocks;
  int lg;               // log2 G: row r of a tile is token r >> lg, head r & (G - 1)
  float qk_scale_log2;  // softmax_scale * log2(e) (* k_scale for a static FP8 pool)
  float v_scale;        // static FP8 pool's V scale (1 for block-scaled pools)
  unsigned int* err;
};

// ---------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (>> 4), descriptor version 1, layout SWIZZLE_128B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// K-major operand: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t kmajor(uint32_t saddr) { return sw128_desc(saddr, 16, 1024); }
// MN-major operand: 64-element blocks of the MN dim 16 KiB apart, 8 K-rows 1024 bytes apart.
__device__ __forceinline__ uint64_t mnmajor(uint32_t saddr) { return sw128_desc(saddr, 16384, 1024); }

// Instruction descriptors: fp32 accumulate, M = N = 128; operand type field
// 0 = binary16 (kind::f16) / E4M3 (kind::f8f6f4), 1 = bfloat16; Q K^T with both
// operands K-major; P V with B MN-major.
constexpr uint32_t kIdescQK = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = (1u << 4) | (1u << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kBf16Types = (1u << 7) | (1u << 10);

// D (TMEM) = A x B (+ D): A in tensor memory (row i in lane i, consecutive K
// elements packed little-endian into 32-bit columns), B in shared memory.
__device__ __forceinline__ void mma_f8_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// The mbarrier gets one arrival once every MMA this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t* w) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
        "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]),
        "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]),
        "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t* w) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};"
      ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
        "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld16u(uint32_t taddr, uint32_t* w) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]),
        "=r"(w[8]), "=r"(w[9]), "=r"(w[10]), "=r"(w[11]), "=r"(w[12]), "=r"(w[13]), "=r"(w[14]), "=r"(w[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// max(a, b, c) in one instruction (the three-input max.f32 of sm_100 and
// later); like fmaxf, a NaN input is ignored.
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Largest of v[0 .. 15]: eight maxima, three deep.
__device__ __forceinline__ float max16(const float* v) {
  const float a = fmax3f(v[0], v[1], v[2]), b = fmax3f(v[3], v[4], v[5]);
  const float c = fmax3f(v[6], v[7], v[8]), d = fmax3f(v[9], v[10], v[11]);
  const float e = fmax3f(v[12], v[13], v[14]);
  return fmaxf(fmax3f(a, b, c), fmax3f(d, e, v[15]));
}

// As mbar_try_wait, but a thread whose phase is not complete may be suspended
// for up to `hint_ns` (woken as soon as the phase completes) instead of the
// hardware's own short limit.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Bounded wait that also gives up as soon as another role has aborted.  Its
// retries sleep (up to 20 us each, woken when the phase completes), so the
// waiting warps leave the issue slots of their scheduler to the warps that
// work, the single MMA-issuing thread above all.  The wait gives up before a
// sleep that could take it past the limit, so a limit shorter than one sleep
// gives up as soon as the first (briefly blocking) test finds the phase
// incomplete.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned int* err) {
  constexpr uint32_t kSleepNs = 20000u;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t limit = pipe_wait_limit();
  const uint64_t t0 = global_ns();
  for (;;) {
    if (*abort_flag) return false;
    if (global_ns() - t0 + kSleepNs > limit) {
      *abort_flag = 1;
      record_error(err, PA_ERR_TIMEOUT);
      return false;
    }
    if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
  }
}

// causal limit of a row: the position of its query token (rows past the
// tile's last token reuse the last one)
__device__ __forceinline__ int qp_of(int pos0, int tl, int n_tok) { return pos0 + min(tl, n_tok - 1); }

template <int OUT>
__device__ __forceinline__ void store_row32(void* out, size_t idx, const float* v, float s) {
  if constexpr (OUT == PA_FP32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + idx);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = make_float4(v[4 * i] * s, v[4 * i + 1] * s, v[4 * i + 2] * s, v[4 * i + 3] * s);
  } else if constexpr (OUT == PA_FP16) {
    uint4* o = reinterpret_cast<uint4*>(static_cast<__half*>(out) + idx);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = make_uint4(pack2<false>(v[8 * i] * s, v[8 * i + 1] * s), pack2<false>(v[8 * i + 2] * s, v[8 * i + 3] * s),
                        pack2<false>(v[8 * i + 4] * s, v[8 * i + 5] * s), pack2<false>(v[8 * i + 6] * s, v[8 * i + 7] * s));
  } else {
    uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + idx);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = make_uint4(pack2<true>(v[8 * i] * s, v[8 * i + 1] * s), pack2<true>(v[8 * i + 2] * s, v[8 * i + 3] * s),
                        pack2<true>(v[8 * i + 4] * s, v[8 * i + 5] * s), pack2<true>(v[8 * i + 6] * s, v[8 * i + 7] * s));
  }
}

template <int KIND, int OUT, bool PSPLIT>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const TcArgs a,
                                                                  const __grid_constant__ CUtensorMap tmk,
                                                                  const __grid_constant__ CUtensorMap tmv) {
  using L = Lay<KIND>;
  constexpr bool F8 = L::kF8, BLK = L::kBlk, BF = L::kBf;
  constexpr int R = L::kRing;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl* ctl = reinterpret_cast<Ctrl*>(sm + L::kData);
  volatile int* abort_flag = &ctl->abort;

  const int qt = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, seq = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = a.q_start[seq];
  const int Cn = a.q_start[seq + 1] - q0;
  // a negative start or a decreasing pair: the sequence is skipped
  if (q0 < 0 || Cn < 0) {
    if (threadIdx.x == 0) record_error(a.err, PA_ERR_BOUNDS);
    return;
  }
  // a chunk longer than the grid covers (max_chunk): its rows past the grid
  // are not written; the CTA of the last tile reports it
  if (qt == (int)gridDim.x - 1 && Cn > ((int)gridDim.x << (7 - a.lg)) && threadIdx.x == 0)
    record_error(a.err, PA_ERR_BOUNDS);
  const int tok_lo = qt << (7 - a.lg);  // a tile holds 128 / G query tokens
  if (tok_lo >= Cn) return;
  const int ctx = a.ctx[seq];
  if (ctx < Cn || ctx > a.max_blocks * 16) {
    if (threadIdx.x == 0) record_error(a.err, PA_ERR_BOUNDS);
    return;
  }
  const int n_tok = min(kRows >> a.lg, Cn - tok_lo);
  const int pos0 = ctx - Cn + tok_lo;  // position of the tile's first query
  const int pos_last = pos0 + n_tok - 1;
  const int npages = pos_last / 16 + 1;
  const int nblk = (npages + 7) / 8;

  if (threadIdx.x == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(&ctl->kv_full[i], 1);
      // FP8: the QK MMAs' commit + the four converter warps; 16-bit: the P V MMAs' commit
      mbar_init(&ctl->kv_empty[i], F8 ? 5 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->vt_full[i], 4);
      mbar_init(&ctl->vt_empty[i], 1);
      mbar_init(&ctl->sc_full[i], 1);
      mbar_init(&ctl->sc_empty[i], 8);
      mbar_init(&ctl->p_full[i], 8);
    }
    mbar_init(&ctl->q_ready, 8);
    mbar_init(&ctl->drain, 1);
    mbar_init(&ctl->xchg, 8);
    mbar_init(&ctl->tail_ready, 1);
    mbar_init(&ctl->tail_done, 4);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(&ctl->tmem)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // A 512-column allocation spans the whole tensor memory, so its base is lane
  // 0, column 0.  FP8 pools take that base as a constant: every tensor-memory
  // operand of the MMA-issuing thread is then an immediate (3% faster on the
  // 8,192-token packet; 16-bit pools measured 2% slower with it, so they keep
  // the allocated address).  A different base is reported and the CTA skips
  // its work.
  const uint32_t tmem_base = ctl->tmem;
  const uint32_t tmem = F8 ? 0u : tmem_base;

  if (F8 && tmem_base != 0) {
    if (threadIdx.x == 0) record_error(a.err, PA_ERR_UNSUPPORTED);
  } else if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    const int32_t* trow = a.tables + (size_t)seq * a.max_blocks;
    const uint64_t policy = l2_evict_first_policy();
    // Lane i holds the table entry (block-scaled: and the tile scales) of page
    // 32 b + i of the current batch of four blocks; the next batch's entries
    // are loaded one batch ahead, so no table load sits between two blocks.
    auto entry = [&](int page) { return page < npages ? trow[page] : 0; };
    int phys = 0, nxt = entry(32 + lane);
    float sk = 1.f, sv = 0.f;
    auto take = [&](int raw, int page) {  // checks the batch's entries and reads their scales
      phys = raw;
      if (page < npages && (raw < 0 || raw >= a.num_blocks)) {
        record_error(a.err, PA_ERR_BOUNDS);
        phys = 0;
      }
      if constexpr (BLK) {
        sk = 1.f;
        sv = 0.f;
        if (page < npages) {
          sk = a.ksc[(size_t)phys * a.Hkv + h];
          sv = a.vsc[(size_t)phys * a.Hkv + h];
        }
      }
    };
    take(entry(lane), lane);
    int issued = 0;
    for (int j = 0; j < nblk; ++j) {
      const int half = j % R, u = j / R;
      const int pb = 8 * (j & 3);  // the block's first page within the batch
      if (j > 0 && pb == 0) {
        take(nxt, 8 * j + lane);
        nxt = entry(8 * j + 32 + lane);
      }
      if (j >= R && !__all_sync(kAll, wait_or_abort(&ctl->kv_empty[half], (u - 1) & 1, abort_flag, a.err))) break;
      const int cnt = min(8, npages - 8 * j);
      if constexpr (BLK) {  // the scales go to buffer j % 2, as the softmax reads them
        const int sb = j & 1;
        if (j >= 2 && !__all_sync(kAll, wait_or_abort(&ctl->sc_empty[sb], ((j >> 1) - 1) & 1, abort_flag, a.err))) break;
        float2 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = make_float2(__shfl_sync(kAll, sk, pb + i), __shfl_sync(kAll, sv, pb + i));
        if (lane == 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) ctl->sc[sb][i] = v[i];
          mbar_arrive(&ctl->sc_full[sb]);
        }
      }
      if (lane == 0) mbar_arrive_expect_tx(&ctl->kv_full[half], (uint32_t)cnt * (F8 ? 4096u : 8192u));
      // each page's copies are issued by the lane that holds its entry, so the
      // block's copies leave in one warp instruction per tile instead of one
      // thread issuing them in turn (a copy landing before lane 0's expect-tx
      // only makes the byte count transiently negative; the phase still waits
      // for that arrival)
      {
        const int i = lane - pb;  // this lane's page within the block
        if (i >= 0 && i < cnt) {
          const int row0 = (phys * a.Hkv + h) * 16;
          uint8_t* kd = sm + L::kKRing + half * L::kSlot + i * 2048;
          uint8_t* vd = sm + L::kVRing + half * L::kSlot + i * 2048;
          if constexpr (F8) {
            tma_load_2d(kd, &tmk, 0, row0, &ctl->kv_full[half], policy);
            tma_load_2d(vd, &tmv, 0, row0, &ctl->kv_full[half], policy);
          } else {  // the two 64-dim (128-byte) halves of each 256-byte row
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              tma_load_2d(kd + hh * 16384, &tmk, 128 * hh, row0, &ctl->kv_full[half], policy);
              tma_load_2d(vd + hh * 16384, &tmv, 128 * hh, row0, &ctl->kv_full[half], policy);
            }
          }
        }
      }
      ++issued;
    }
    // no copy may still target shared memory when the CTA exits
    if (lane == 0)
      for (int j = max(0, issued - R); j < issued; ++j)
        if (!mbar_wait(&ctl->kv_full[j % R], (j / R) & 1)) record_error(a.err, PA_ERR_TIMEOUT);
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0 && wait_or_abort(&ctl->q_ready, 0, abort_flag, a.err)) {
      // Descriptors are computed once: moving an operand by X bytes adds X / 16
      // to the descriptor's start-address field (shared addresses stay below
      // 256 KiB, so the field never carries), which keeps the issuing thread's
      // work between two MMAs to a few instructions.
      const uint64_t kdesc0 = kmajor(smem_addr(sm + L::kKRing));
      const uint64_t vdesc0 = mnmajor(smem_addr(sm + (F8 ? L::kVT : L::kVRing)));
      // S(j) = Q K(j)^T into S buffer j % 2
      auto issue_qk = [&](int j) {
        const int sb = j & 1;
        if constexpr (!F8)
          if (j == nblk - 1) mbar_arrive(&ctl->tail_ready);  // its pages have landed
        const uint64_t kd = kdesc0 + (uint64_t)((j % R) * (L::kSlot >> 4));
        if constexpr (F8) {
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f8_ts(tmem + sb * 128, tmem + (t ? kQLoCol : kQHiCol) + 8 * k, kd + 2 * k, kIdescQK,
                        (uint32_t)(t | k));
        } else {  // 16 dims per MMA: dim half k / 4, 32 bytes into its rows
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_f16_ts(tmem + sb * 128, tmem + kQHiCol + 8 * k, kd + (k >> 2) * (16384 >> 4) + (k & 3) * 2,
                       kIdescQK | (BF ? kBf16Types : 0u), (uint32_t)k);
        }
        mma_commit(&ctl->s_full[sb]);
        if constexpr (F8) mma_commit(&ctl->kv_empty[j % R]);  // K is read; V was converted
      };
      // Order: S(0), S(1), then per block i: O += P(i) V(i) and S(i + 2) right
      // behind it (its P lives in S buffer i % 2; the MMAs run in issue order).
      // The tensor pipe thus runs P V and the next Q K^T back to back while the
      // softmax works on block i + 1, whose S was computed one step earlier.
      bool run = true;
      for (int j = 0; j < 2 && j < nblk && run; ++j) {
        run = wait_or_abort(&ctl->kv_full[j % R], (j / R) & 1, abort_flag, a.err);
        if (run) {
          tc_fence_after();
          issue_qk(j);
        }
      }
      if constexpr (F8) {
        // FP8 pools (a two-slot ring): blocks in pairs, so every operand's
        // slot and buffer is a compile-time parity and all 24 shared-memory
        // descriptors live in registers (the tensor-memory addresses are the
        // base plus constants).  The issuing thread shares its scheduler with
        // three busy warps, so its instructions between MMAs, not the tensor
        // pipe, had set the pace: 5% faster this way.  Same MMAs in the same
        // order as the loop below.
        static_assert(!F8 || R == 2, "the paired loop assumes a two-slot ring");
        uint64_t qkb[2][4], pvb[2][8];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
#pragma unroll
          for (int k = 0; k < 4; ++k) qkb[p][k] = kdesc0 + (uint64_t)(p * (L::kSlot >> 4) + 2 * k);
#pragma unroll
          for (int k = 0; k < 8; ++k) pvb[p][k] = vdesc0 + (uint64_t)(p * (32768 >> 4) + k * (2048 >> 4));
        }
        auto step = [&](auto par, int i) -> bool {
          constexpr int P = decltype(par)::value;  // i % 2
          if (!wait_or_abort(&ctl->p_full[P], (i >> 1) & 1, abort_flag, a.err)) return false;
          if (!wait_or_abort(&ctl->vt_full[P], (i >> 1) & 1, abort_flag, a.err)) return false;
          tc_fence_after();
#pragma unroll
          for (int part = 0; part < (PSPLIT ? 2 : 1); ++part)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_f16_ts(tmem + kOCol, tmem + P * 128 + 32 * (k >> 1) + 16 * part + 8 * (k & 1), pvb[P][k],
                         kIdescPV, (uint32_t)(i | k | part));
          mma_commit(&ctl->vt_empty[P]);
          if (i + 2 < nblk) {  // S(i + 2) into S buffer P, from ring slot P
            if (!wait_or_abort(&ctl->kv_full[P], ((i + 2) >> 1) & 1, abort_flag, a.err)) return false;
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f8_ts(tmem + P * 128, tmem + (t ? kQLoCol : kQHiCol) + 8 * k, qkb[P][k], kIdescQK,
                          (uint32_t)(t | k));
            mma_commit(&ctl->s_full[P]);
            mma_commit(&ctl->kv_empty[P]);
          }
          return true;
        };
        for (int i = 0; i < nblk && run; i += 2) {
          run = step(std::integral_constant<int, 0>{}, i);
          if (run && i + 1 < nblk) run = step(std::integral_constant<int, 1>{}, i + 1);
        }
        run = false;  // the loop below is for 16-bit pools
      }
      for (int i = 0; i < nblk && run; ++i) {
        const int vb = i & 1;
        if (!wait_or_abort(&ctl->p_full[i & 1], (i >> 1) & 1, abort_flag, a.err)) break;
        if constexpr (F8) {
          if (!wait_or_abort(&ctl->vt_full[vb], (i >> 1) & 1, abort_flag, a.err)) break;
        } else {
          if (i == nblk - 1 && !wait_or_abort(&ctl->tail_done, 0, abort_flag, a.err)) break;
        }
        tc_fence_after();
        // B: the binary16 V block (FP8 pools) or the V ring slot itself (16-bit pools)
        const uint64_t vd = vdesc0 + (uint64_t)(F8 ? vb * (32768 >> 4) : (i % R) * (L::kSlot >> 4));
#pragma unroll
        for (int part = 0; part < (PSPLIT ? 2 : 1); ++part)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_f16_ts(tmem + kOCol, tmem + vb * 128 + 32 * (k >> 1) + 16 * part + 8 * (k & 1),
                       vd + k * (2048 >> 4), kIdescPV | (BF ? kBf16Types : 0u), (uint32_t)(i | k | part));
        if constexpr (F8) mma_commit(&ctl->vt_empty[vb]);
        else mma_commit(&ctl->kv_empty[i % R]);  // K and V of block i are read
        if (i + 2 < nblk) {
          // S(i + 2) goes into the TMEM columns P V(i) reads P(i) from.  The
          // MMAs of one thread run in issue order, so Q K^T(i + 2) is issued
          // right behind P V(i) without waiting for it to finish.
          if (!wait_or_abort(&ctl->kv_full[(i + 2) % R], ((i + 2) / R) & 1, abort_flag, a.err)) break;
          tc_fence_after();
          issue_qk(i + 2);
        }
      }
      // every MMA issued above has finished before O is read and TMEM released
      mma_commit(&ctl->drain);
      if (!mbar_wait(&ctl->drain, 0)) record_error(a.err, PA_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp < 4 || warp >= 12) {
    // ---------------------------------------------------------- V to binary16
    // four warps, one per scheduler; consecutive lanes take consecutive keys of
    // one 16-byte chunk, so each 8-lane phase of a 16-byte access covers 8
    // distinct (swizzled) chunks
    const int ct = 32 * (warp < 4 ? warp - 2 : warp - 10) + lane;  // 0 .. 127
    if constexpr (!F8) {
      // 16-bit pools: nothing to convert, but V is read in place, so the rows
      // of the last block past the tile's last query (stale slots of its last
      // page, pages not loaded) are zeroed: P is 0 there, and 0 x NaN is not.
      // The MMA warp signals once that block's copies have landed (its ring
      // slot is used for nothing else afterwards, so kv_full stays complete).
      const int j = nblk - 1;
      bool go = __all_sync(kAll, wait_or_abort(&ctl->tail_ready, 0, abort_flag, a.err));
      go = go && __all_sync(kAll, wait_or_abort(&ctl->kv_full[j % R], (j / R) & 1, abort_flag, a.err));
      if (go) {
        const int nvalid = pos_last + 1 - 128 * j;  // 1 .. 128
        uint8_t* vr = sm + L::kVRing + (j % R) * L::kSlot;
        for (int idx = ct; idx < (128 - nvalid) * 16; idx += 128) {  // 16 chunks of 16 B per key
          const int key = nvalid + (idx >> 4), c = idx & 15;
          *reinterpret_cast<uint4*>(vr + (c >> 3) * 16384 + key * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->tail_done);
      }
    }
    for (int j = 0; j < (F8 ? nblk : 0); ++j) {
      const int slot = j % R, half = j & 1, u = j >> 1;  // ring slot; binary16 V buffer
      if (!__all_sync(kAll, wait_or_abort(&ctl->kv_full[slot], (j / R) & 1, abort_flag, a.err))) break;
      if (j >= 2 && !__all_sync(kAll, wait_or_abort(&ctl->vt_empty[half], (u - 1) & 1, abort_flag, a.err))) break;
      const int nvalid = min(128, pos_last + 1 - 128 * j);  // keys past the last query: zero
      const uint8_t* vr = sm + L::kVRing + slot * L::kSlot;
      uint8_t* vt = sm + L::kVT + half * 32768;
#pragma unroll 4
      for (int it = 0; it < 8; ++it) {
        const int idx = ct + 128 * it, key = idx & 127, ch = idx >> 7;
        uint4 w = make_uint4(0, 0, 0, 0);
        if (key < nvalid) w = lds128(vr + (key >> 4) * 2048 + (key & 15) * 128 + ((ch ^ (key & 7)) << 4));
        const uint32_t cw[4] = {w.x, w.y, w.z, w.w};
        uint32_t hv[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          e4m3x4_to_f16x2x2(cw[q], hv[2 * q], hv[2 * q + 1]);
        }
        uint8_t* row = vt + (ch >> 2) * 16384 + key * 128;
        const int c0 = (ch & 3) * 2;
        *reinterpret_cast<uint4*>(row + ((c0 ^ (key & 7)) << 4)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (key & 7)) << 4)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->vt_full[half]);
        mbar_arrive(&ctl->kv_empty[slot]);
      }
    }
  } else {
    // ---------------------------------------------------------- softmax rows
    // Two threads per row: row r (= G * query token + head) in TMEM lane r; the
    // thread of half hf takes keys 64 hf .. 64 hf + 63 of every block (two
    // 32-column chunks), O columns 64 hf .. 64 hf + 63, and Q dims 64 hf ...
    // The halves exchange partials through shared memory, one xchg phase each
    // (Q amax, then every block's max, then the row sum).  Every softmax warp
    // runs every block and arrives at every phase even after an abort (its
    // waits then return at once), so the phases of xchg stay in step.
    const int sw = warp - 4, hf = sw >> 2;
    const int r = (sw & 3) * 32 + lane;
    const int tl = r >> a.lg, hh = r & ((1 << a.lg) - 1);
    const bool row_valid = tl < n_tok;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    int xk = 0;  // next xchg phase
    bool ok = true;
    auto exchange = [&](float mine, float& lo_half, float& hi_half) {
      ctl->xbuf[xk & 1][r][hf] = mine;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->xchg);
      ok = __all_sync(kAll, (ok && wait_or_abort(&ctl->xchg, xk & 1, abort_flag, a.err)));
      lo_half = ctl->xbuf[xk & 1][r][0];
      hi_half = ctl->xbuf[xk & 1][r][1];
      ++xk;
    };

    // Q: scaled by a power of two (max |q| of the row in [128, 256)) and split
    // into two E4M3 terms, stored in TMEM as the A operand of S = Q K^T
    float row_scale = a.qk_scale_log2;
    {
      uint32_t qw[32];  // this half's 64 16-bit values, two per word
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + ((size_t)(q0 + tok_lo + tl) * a.Hq + ((size_t)h << a.lg) + hh) * kD + 64 * hf);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = row_valid ? src[c] : make_uint4(0, 0, 0, 0);
        qw[4 * c] = v.x;
        qw[4 * c + 1] = v.y;
        qw[4 * c + 2] = v.z;
        qw[4 * c + 3] = v.w;
      }
      float am = 0.f;
      if constexpr (F8) {
#pragma unroll
        for (int w = 0; w < 32; ++w)
          am = fmaxf(am, fmaxf(fabsf(bf16_bits_to_float(qw[w] & 0xFFFFu)), fabsf(bf16_bits_to_float(qw[w] >> 16))));
      }
      float a0, a1;
      exchange(am, a0, a1);  // (16-bit pools exchange nothing useful; the phase keeps step)
      if constexpr (!F8) {
        // 16-bit pools: Q itself is the A operand, exact; a negative score scale
        // flips its signs so the per-row factor is positive
        row_scale = fabsf(a.qk_scale_log2);
        if (a.qk_scale_log2 < 0.f) {
#pragma unroll
          for (int w = 0; w < 32; ++w) qw[w] ^= 0x80008000u;
        }
        tmem_st32u(trow + kQHiCol + 32 * hf, qw);
      } else {
      const float amax = fmaxf(a0, a1);
      int ex = 0;
      if (amax > 0.f) frexpf(amax, &ex);
      // a negative score scale goes into q, so the per-row factor is positive
      const float sgn = a.qk_scale_log2 < 0.f ? -1.f : 1.f;
      const float qs = sgn * (amax > 0.f ? ldexpf(1.f, 8 - ex) : 1.f);
      row_scale = fabsf(a.qk_scale_log2) * (amax > 0.f ? ldexpf(1.f, ex - 8) : 1.f);
      uint32_t qhi[16], qlo[16];  // 4 dims per word, dim order
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint32_t w0 = qw[2 * c], w1 = qw[2 * c + 1];
        const float2 x01 = make_float2(bf16_bits_to_float(w0 & 0xFFFFu) * qs, bf16_bits_to_float(w0 >> 16) * qs);
        const float2 x23 = make_float2(bf16_bits_to_float(w1 & 0xFFFFu) * qs, bf16_bits_to_float(w1 >> 16) * qs);
        const uint32_t h01 = __nv_cvt_float2_to_fp8x2(x01, __NV_SATFINITE, __NV_E4M3);
        const uint32_t h23 = __nv_cvt_float2_to_fp8x2(x23, __NV_SATFINITE, __NV_E4M3);
        const float2 d01 = unpack2<false>(e4m3x2_to_f16x2(h01));
        const float2 d23 = unpack2<false>(e4m3x2_to_f16x2(h23));
        const uint32_t l01 = __nv_cvt_float2_to_fp8x2(make_float2(x01.x - d01.x, x01.y - d01.y), __NV_SATFINITE, __NV_E4M3);
        const uint32_t l23 = __nv_cvt_float2_to_fp8x2(make_float2(x23.x - d23.x, x23.y - d23.y), __NV_SATFINITE, __NV_E4M3);
        qhi[c] = (h01 & 0xFFFFu) | (h23 << 16);
        qlo[c] = (l01 & 0xFFFFu) | (l23 << 16);
      }
      tmem_st16u(trow + kQHiCol + 16 * hf, qhi);
      tmem_st16u(trow + kQLoCol + 16 * hf, qlo);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->q_ready);
    }
    // Masked keys hold -inf and meet the score factor in the exponent's
    // multiply, where a zero factor (softmax_scale 0, or a page of zero K
    // scale) would give -inf * 0 = NaN.  Every factor is kept at or above the
    // smallest normal float: scores then round to ~0 in log2 units and the
    // visible keys weigh the same, which is what a zero scale asks for.
    constexpr float kMinFactor = 1.17549435e-38f;
    row_scale = fmaxf(row_scale, kMinFactor);

    float m = -INFINITY, l = 0.f, vref = 0.f;
    for (int j = 0; j < nblk; ++j) {
      const int sb = j & 1, u = j >> 1;
      float ov = 1.f, vinv = 1.f;  // factor for this row's O accumulator; 1 / vref
      if constexpr (BLK) {  // V weights are taken relative to the largest V scale seen (<= 1)
        ok = __all_sync(kAll, ok && wait_or_abort(&ctl->sc_full[sb], u & 1, abort_flag, a.err));
        float vb = vref;
#pragma unroll
        for (int i = 0; i < 8; ++i) vb = fmaxf(vb, ctl->sc[sb][i].y);
        if (vb > vref) {
          ov = vref / vb;
          vref = vb;
        }
        vinv = vref > 0.f ? 1.f / vref : 0.f;
      }
      ok = __all_sync(kAll, ok && wait_or_abort(&ctl->s_full[sb], u & 1, abort_flag, a.err));
      // Scores in log2 units are s * f_page, f_page > 0.  The thread's 64 scores
      // are read from TMEM once and kept in registers through the max exchange
      // (the block max first, then the exponentials); the causal mask runs only
      // on blocks that reach the tile's first query.
      const int key0 = 128 * j;
      const bool diag = key0 + 127 > pos0;
      const uint32_t sbase = trow + sb * 128;
      float pf[2][2];  // the score factor of each of the thread's four pages
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int hp = 0; hp < 2; ++hp)
          pf[cc][hp] = BLK ? fmaxf(row_scale * ctl->sc[sb][2 * (2 * hf + cc) + hp].x, kMinFactor) : row_scale;
      float mh = -INFINITY;
      float sv[2][32];  // this thread's 64 scores of the block, read from TMEM once
      if (ok) {
        tc_fence_after();
        tmem_ld32(sbase + 32 * (2 * hf), sv[0]);
        tmem_ld32(sbase + 32 * (2 * hf + 1), sv[1]);
        tmem_wait_ld();
        float pm[2][2];  // each page's largest raw score
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float* v = sv[cc];
          if (diag) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (key0 + 32 * (2 * hf + cc) + e > qp_of(pos0, tl, n_tok)) v[e] = -INFINITY;
          }
          pm[cc][0] = max16(v);
          pm[cc][1] = max16(v + 16);
        }
        if constexpr (BLK)
          mh = fmaxf(fmax3f(pm[0][0] * pf[0][0], pm[0][1] * pf[0][1], pm[1][0] * pf[1][0]), pm[1][1] * pf[1][1]);
        else  // one positive factor: the largest product is the largest score times it
          mh = fmaxf(fmax3f(pm[0][0], pm[0][1], pm[1][0]), pm[1][1]) * row_scale;
      }
      float m0, m1;
      exchange(mh, m0, m1);
      const float mx = fmaxf(m0, m1);
      if (mx > m + 8.f) {  // the first visible block, or a max that grew by more than 2^8
        const float alpha = fast_exp2(m - mx);
        l *= alpha;
        ov *= alpha;
        m = mx;
      }
      // O is rescaled once the previous block's P V is done (rarely needed),
      // seen through the barrier committed right behind that P V: the binary16
      // V buffer's (FP8) or the ring slot's (16-bit) release.  Phase distance:
      // s_full(j) was committed after Q K^T(j), issued after P V(j - 2), and a
      // commit tracks every earlier MMA of the thread, so that barrier's phase
      // before P V(j - 1)'s is complete; its phase after needs P(j + 1) or
      // later, which is not stored yet.  So the awaited phase is pending or just
      // completed, never mistaken.
      if (ok && j > 0 && __any_sync(kAll, ov != 1.f)) {
        ok = __all_sync(kAll, F8 ? wait_or_abort(&ctl->vt_empty[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, a.err)
                                 : wait_or_abort(&ctl->kv_empty[(j - 1) % R], ((j - 1) / R) & 1, abort_flag, a.err));
        if (ok) {
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {  // 16 columns at a time (the scores are live)
            uint32_t o[16];
            const uint32_t oc = trow + kOCol + 64 * hf + 16 * cc;
            tmem_ld16u(oc, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * ov);
            tmem_st16u(oc, o);
          }
          tmem_wait_st();
        }
      }
      // P in binary16 over the chunk's own S columns: keys 32c .. 32c+31 go to
      // columns 32c .. 32c+15 (the low part, fp32 mode, to 32c+16 .. 32c+31)
      if (ok) {
        float rs = 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * hf + cc;
          float* v = sv[cc];  // masked in the first pass
#pragma unroll
          for (int hp = 0; hp < 2; ++hp) {
            // two keys per packed multiply-add and add; the sums keep the
            // order of four running sums over keys e = 0, 1, 2, 3 (mod 4)
            const float2 f2 = make_float2(pf[cc][hp], pf[cc][hp]), nm = make_float2(-m, -m);
            const float vm = BLK ? ctl->sc[sb][2 * c + hp].y * vinv : 1.f;
            const float2 vm2 = make_float2(vm, vm);
            float2 t01 = make_float2(0.f, 0.f), t23 = t01;
            float* x = v + 16 * hp;
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
              const float2 za = __ffma2_rn(make_float2(x[e], x[e + 1]), f2, nm);
              const float2 zb = __ffma2_rn(make_float2(x[e + 2], x[e + 3]), f2, nm);
              float2 pa = make_float2(fast_exp2(za.x), fast_exp2(za.y));
              float2 pb = make_float2(fast_exp2(zb.x), fast_exp2(zb.y));
              t01 = __fadd2_rn(t01, pa);
              t23 = __fadd2_rn(t23, pb);
              if constexpr (BLK) {
                pa = __fmul2_rn(pa, vm2);
                pb = __fmul2_rn(pb, vm2);
              }
              x[e] = pa.x;
              x[e + 1] = pa.y;
              x[e + 2] = pb.x;
              x[e + 3] = pb.y;
            }
            rs += (t01.x + t01.y) + (t23.x + t23.y);
          }
          uint32_t ph[16], pl[16];  // in V's type: bfloat16 for bfloat16 pools, else binary16
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            ph[e] = pack2<BF>(v[2 * e], v[2 * e + 1]);
            if constexpr (PSPLIT) {
              const float2 hv = unpack2<BF>(ph[e]);
              pl[e] = pack2<BF>(v[2 * e] - hv.x, v[2 * e + 1] - hv.y);
            }
          }
          tmem_st16u(sbase + 32 * c, ph);
          if constexpr (PSPLIT) tmem_st16u(sbase + 32 * c + 16, pl);
        }
        l += rs;
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (BLK) mbar_arrive(&ctl->sc_empty[sb]);
        mbar_arrive(&ctl->p_full[sb]);
      }
    }
    // output rows: O / l (times the V scale), once every MMA is done (the
    // one-phase drain barrier, committed behind the last P V)
    float l0, l1;
    exchange(l, l0, l1);
    const float L = l0 + l1;
    ok = __all_sync(kAll, ok && wait_or_abort(&ctl->drain, 0, abort_flag, a.err));
    if (ok) {
      tc_fence_after();
      const float sc = L > 0.f ? (BLK ? vref : a.v_scale) / L : 0.f;
      const size_t orow = ((size_t)(q0 + tok_lo + tl) * a.Hq + ((size_t)h << a.lg) + hh) * kD + 64 * hf;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        float o[32];
        tmem_ld32(trow + kOCol + 64 * hf + 32 * cc, o);
        tmem_wait_ld();
        if (row_valid) store_row32<OUT>(a.out, orow + 32 * cc, o, sc);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols) : "memory");
  }
}

struct TcInfo {
  const void* fn;
  int smem;
  bool configured[128];
};

template <int KIND, int OUT, bool PSPLIT>
TcInfo& tc_info() {
  static TcInfo ti = {reinterpret_cast<const void*>(&prefill_tc_kernel<KIND, OUT, PSPLIT>), Lay<KIND>::kSmem, {}};
  return ti;
}

template <int KIND, int OUT, bool PSPLIT>
cudaError_t tc_launch(const TcArgs& a, const CUtensorMap* tk, const CUtensorMap* tv, int tiles, int S,
                      cudaStream_t st) {
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  TcInfo& ti = tc_info<KIND, OUT, PSPLIT>();
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    if (!ti.configured[dev]) {
      e = cudaFuncSetAttribute(ti.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ti.smem);
      if (e != cudaSuccess) return e;
      ti.configured[dev] = true;
    }
  }
  prefill_tc_kernel<KIND, OUT, PSPLIT><<<dim3(tiles, a.Hkv, S), kThreads, ti.smem, st>>>(a, *tk, *tv);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const pa_pool* pool, int n_q_heads, int out_dtype) {
  const pa_pool_desc& d = pool->desc;
  if (d.head_dim != kD || n_q_heads % d.n_kv_heads != 0) return false;
  const int G = n_q_heads / d.n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  switch (d.kv_dtype) {
    case PA_FP8_E4M3:
    case PA_FP8_E4M3_BLOCK:
    case PA_BF16:
      return out_dtype == PA_BF16 || out_dtype == PA_FP32;
    case PA_FP16:
      return out_dtype == PA_FP16 || out_dtype == PA_FP32;
    default:
      return false;
  }
}

int prefill_tc(pa_pool* pool, int layer, void* out, int out_dtype, const void* q, const int32_t* q_start,
               const int32_t* tables, int max_blocks, const int32_t* ctx, int S, int n_q_heads,
               int max_chunk, float softmax_scale, unsigned int* err, cudaStream_t st) {
  const pa_pool_desc& d = pool->desc;
  const bool f8 = d.kv_dtype == PA_FP8_E4M3 || d.kv_dtype == PA_FP8_E4M3_BLOCK;
  const CUtensorMap_st *tk = nullptr, *tv = nullptr;
  int rc = f8 ? layer_maps(pool, layer, &tk, &tv) : layer_half_maps(pool, layer, &tk, &tv);
  if (rc) return rc;
  TcArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.out = out;
  a.q_start = q_start;
  a.ctx = ctx;
  a.tables = tables;
  a.ksc = pool->block_scaled ? layer_scales(pool, pool->k, layer) : nullptr;
  a.vsc = pool->block_scaled ? layer_scales(pool, pool->v, layer) : nullptr;
  a.max_blocks = max_blocks;
  a.Hq = n_q_heads;
  a.Hkv = d.n_kv_heads;
  a.num_blocks = d.num_blocks;
  const bool static_fp8 = d.kv_dtype == PA_FP8_E4M3;
  a.qk_scale_log2 = softmax_scale * 1.4426950408889634f * (static_fp8 ? d.k_scale : 1.f);
  a.v_scale = static_fp8 ? d.v_scale : 1.f;
  a.err = err;
  const int G = n_q_heads / d.n_kv_heads;
  a.lg = G == 8 ? 3 : G == 4 ? 2 : G == 2 ? 1 : 0;
  const int tok = kRows >> a.lg;
  const int tiles = (max_chunk + tok - 1) / tok;
  const bool f32 = out_dtype == PA_FP32;
  cudaError_t e;
  switch (d.kv_dtype) {
    case PA_FP8_E4M3:
      e = f32 ? tc_launch<K_E4M3, PA_FP32, true>(a, tk, tv, tiles, S, st)
              : tc_launch<K_E4M3, PA_BF16, false>(a, tk, tv, tiles, S, st);
      break;
    case PA_FP8_E4M3_BLOCK:
      e = f32 ? tc_launch<K_E4M3B, PA_FP32, true>(a, tk, tv, tiles, S, st)
              : tc_launch<K_E4M3B, PA_BF16, false>(a, tk, tv, tiles, S, st);
      break;
    case PA_BF16:  // P in bfloat16 carries 8 bits: always split into two parts
      e = f32 ? tc_launch<K_BF16, PA_FP32, true>(a, tk, tv, tiles, S, st)
              : tc_launch<K_BF16, PA_BF16, true>(a, tk, tv, tiles, S, st);
      break;
    default:
      e = f32 ? tc_launch<K_F16, PA_FP32, true>(a, tk, tv, tiles, S, st)
              : tc_launch<K_F16, PA_FP16, false>(a, tk, tv, tiles, S, st);
      break;
  }
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "prefill (tcgen05) launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

int prefill_tc_set_wait_limit(unsigned long long ns) { return (int)set_pipe_wait_limit_here(ns); }

}  // namespace pa
