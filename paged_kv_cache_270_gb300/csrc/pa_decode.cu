// pa_decode.cu -- paged decode attention for sm_103a.
//
// One query token per sequence attends to its whole paged history: the
// kernel takes the block table as an extra input and gathers each 16-token
// page of keys and values by indirection instead of slicing a contiguous slab
// ("Capítulo 8 -- Gestión de caché KV de nueva generación", section 8.1).
// Pages may hold FP8 E4M3 codes with a static per-tensor scale or with a scale
// per (block, kv head) tile, dequantised as they are used ("Optimización de KV
// Cache con PagedAttention y Cuantización FP8 para Contextos Largos (128K)",
// sections 4 and 8, static calibration and dynamic scaling).  Long contexts (up to
// the 128K of that page's title) are split along their pages; a second kernel
// merges the partial softmax states.
//
// Kernel design (not from the pages; they give none):
//  * grid = (split, kv head, sequence); 5 warps per CTA.
//  * Warp 4 is the producer: it reads the sequence's block-table entries 32 at a
//    time (one coalesced load) and issues, per page, two TMA tensor copies (the
//    contiguous K tile and V tile of this kv head, 16 rows of head_dim
//    elements) into an 8-stage shared-memory ring, completing on an mbarrier.
//    Rows of 128 or 256 bytes are written with the TMA's 128-byte swizzle, so
//    the consumers' 16-byte shared-memory reads below are bank-conflict free.
//    The tiles are streamed once, so they carry an L2 evict-first hint.
//  * Warps 0..3 consume whole pages round-robin in logical order.  The whole
//    grouped-query group (G <= 8 query heads sharing this kv head) is resident,
//    so every KV byte is read from HBM exactly once per decode.
//  * S^T = K_page * Q^T is one m16n8k16 tensor-core MMA per 16 dims
//    (M = 16 tokens of the page, N = 8 query heads, fp32 accumulate); the
//    online softmax runs in the log2 domain on the accumulator fragment; P is
//    transposed in registers (movmatrix) into the B operand of
//    O^T += V_page^T * P^T (M = 16 dims per MMA, K = the 16 tokens).
//    Any permutation of the head dimension that Q and K share leaves q.k
//    unchanged, so each thread loads a contiguous 16-byte run of a K row and
//    the matching Q run.  V comes through a transposed ldmatrix, which hands
//    each thread consecutive tokens of one V column: token pairs for 16-bit
//    pools, four tokens for FP8 pools, whose tokens are then taken in an order
//    that makes those four the A operand's two pairs (K rows follow the same
//    order).  Rows narrower than 128 bytes (d = 64 FP8) keep byte permutes.
//  * FP8 codes convert exactly to binary16, two at a time from the 16-bit
//    halves of a register (reaching the upper pair by shifting the word would
//    cost an instruction per conversion); q (bfloat16) is rescaled by a power
//    of two so the group's largest |q| lands in [2^14, 2^15) before rounding to
//    binary16, and the scale is folded back into the softmax exponent.  For
//    bfloat16 pools (and in fp32-output mode) P is split into a high and a low
//    16-bit part, two MMAs, so P carries ~16 significant bits.
//  * Per-tile scales (block-scaled pools) ride with the page: the producer reads
//    them next to the table entries and hands them over in shared memory; the
//    K scale joins the softmax exponent's factor, the V scale weights P
//    relative to the largest V scale seen so far (kept <= 1 for 16-bit P).
//  * Accumulation follows logical page order within each warp and a fixed warp
//    order in the merge, so the result is bit-identical under any relabelling
//    of physical blocks.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "pa_device.cuh"

namespace pa {

enum KvKind { KV_F16 = 0, KV_BF16 = 1, KV_E4M3 = 2, KV_E4M3B = 4 };  // KV_E4M3B: scale per tile
enum OutKind { OUT_F16 = 0, OUT_BF16 = 1, OUT_F32 = 3 };

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr unsigned kFull = 0xffffffffu;

template <int KV, int D>
struct Cfg {
  static constexpr bool kFp8 = (KV == KV_E4M3) || (KV == KV_E4M3B);
  static constexpr bool kBlockScaled = (KV == KV_E4M3B);
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;    // one token row of a tile
  static constexpr int kTile = 16 * kRowBytes;   // bytes of one (block, kv head) tile
  // Rows of 128 or 256 bytes are loaded with 128-byte TMA swizzling, which
  // makes every shared-memory read of the consumers below bank-conflict free.
  static constexpr bool kSwizzle = (kRowBytes % 128) == 0;
  static constexpr int kTmaRank = kRowBytes == 256 ? 3 : 2;
  static constexpr int kStages = 8;
  // Consumer warp w takes pages w, w + 4, ...; with a stage count that is a
  // multiple of the warp count, the previous page of a stage is the same
  // warp's, so a warp waits on a full barrier at most one phase behind (the
  // parity wait cannot tell phases further apart).
  static_assert(kStages % kConsumerWarps == 0, "stages must be a multiple of the consumer warps");
  static constexpr int kStageBytes = 2 * kTile;  // K tile + V tile
  static constexpr int kRingBytes = kStages * kStageBytes;
  // merge area: per warp, 8 heads x (D + 4) floats (the pad spreads a warp's
  // stores over all banks) plus (m, l) per head
  static constexpr int kMergeStride = D + 4;
  static constexpr int kMergeBytes = kConsumerWarps * 8 * (kMergeStride + 2) * 4;
  static constexpr int kDataBytes = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
  static constexpr int kAlign = 1024;  // a 128-byte-swizzled TMA destination is 1 KiB aligned
  // FP8 pools keep the query fragments in shared memory instead of 16 registers
  // per thread ([warp][D/16 pairs][32 lanes] x 8 bytes), which lets five CTAs
  // share an SM; 16-bit pools are limited by their ring size anyway.
  static constexpr bool kQInSmem = kFp8;
  static constexpr int kQBytes = kQInSmem ? kConsumerWarps * (D / 16) * 32 * 8 : 0;
  // block-scaled pools: the (K, V) scales of the page in each stage
  static constexpr int kScaleBytes = kBlockScaled ? kStages * 8 : 0;
  static constexpr int kSmem = kDataBytes + 2 * kStages * 8 + kQBytes + kScaleBytes + kAlign;
  // register budget, in CTAs per SM (16-bit pools: what their ring size allows).
  // Block-scaled FP8 spills a little at five, so it has a second build for four
  // (kMinBlocksLow), taken by launches that put at most four CTAs on an SM.
  static constexpr int kMinBlocks = kQInSmem ? 5 : (D == 128 ? 3 : 4);
  static constexpr int kMinBlocksLow = kBlockScaled ? 4 : kMinBlocks;
  static constexpr bool kMmaBf16 = (KV == KV_BF16);
  static_assert(kStageBytes % kAlign == 0 || !kSwizzle, "tiles must stay 1 KiB aligned");
};

// The balanced schedule gives every CTA at least this many pages.
constexpr int kMinPagesPerCta = 8;

// Fixed splits: how a sequence's pages are cut.  Uniform: split k covers pages
// [k pps, (k + 1) pps).  Guided (the automatic layout of launches of several
// waves): split k covers [b[k], b[k + 1]), sizes falling geometrically, and
// the split index is the slowest grid dimension, so the block scheduler hands
// out every sequence's first (largest) split first and the small last splits
// last: the CTAs still running as the grid drains are short ones.
constexpr int kGuidedSplits = 8;
struct SplitLayout {
  int splits, pps;
  int guided;
  int b[kGuidedSplits + 1];
};

struct DecodeArgs {
  const uint16_t* q;     // [S][Hq][D]
  void* out;             // [S][Hq][D]
  // split partials.  Fixed splits: [S][Hq][splits][D] and [S][Hq][splits][2]
  // (m in log2 units, l).  Balanced schedule: [2 * ctas][G][D] and [2 * ctas][G][2].
  float* ws_o;
  float* ws_ml;
  int4* jobs;            // balanced schedule: [ctas] merge jobs (sequence, kv head, last CTA, slot)
  const int32_t* tables;
  const int32_t* ctx;
  int max_blocks;
  int S, Hq, Hkv, G, num_blocks;
  int splits, pages_per_split;  // fixed splits (uniform layout)
  SplitLayout sl;               // fixed splits: the layout (uniform or guided)
  int ctas;                     // balanced schedule: CTAs of the launch
  float qk_scale_log2;  // softmax_scale * log2(e) (* k_scale for FP8)
  float v_scale;        // 1 for 16-bit and block-scaled pools
  const float* ksc;     // block-scaled pools: this layer's scales [num_blocks][Hkv]
  const float* vsc;
  unsigned int* err;
};

__device__ __forceinline__ int clamp_ctx(int c, int max_blocks) { return c < 0 ? 0 : min(c, max_blocks * 16); }

// Pages [pb, pe) of split k (the guided bounds are read with constant indices,
// so the layout stays in the parameter space).
__device__ __forceinline__ void split_pages(const SplitLayout& L, int k, int& pb, int& pe) {
  if (L.guided) {
    pb = 0;
    pe = 0;
#pragma unroll
    for (int i = 0; i < kGuidedSplits; ++i)
      if (i == k) {
        pb = L.b[i];
        pe = L.b[i + 1];
      }
  } else {
    pb = k * L.pps;
    pe = pb + L.pps;
  }
}
__device__ __forceinline__ int first_split_pages(const SplitLayout& L) { return L.guided ? L.b[1] : L.pps; }


// Exclusive prefix sum over the CTA's threads (every thread must call it);
// `total` receives the sum over all of them.
template <int NTHREADS>
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* warp_sums,
                                                          long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  long long before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < NTHREADS / 32; ++w) {
    const long long s = warp_sums[w];
    before += w < warp ? s : 0;
    total += s;
  }
  return before + x - v;
}

template <int OUT>
__device__ __forceinline__ void store_out(void* out, size_t idx, float v) {
  if constexpr (OUT == OUT_F32) {
    static_cast<float*>(out)[idx] = v;
  } else if constexpr (OUT == OUT_BF16) {
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(out)[idx] = __float2half_rn(v);
  }
}

// Loads the K or V tile of `row0` (= (block * Hkv + head) * 16) through the map.
template <int RANK>
__device__ __forceinline__ void load_tile(void* dst, const CUtensorMap* map, int row0,
                                          uint64_t* bar, uint64_t policy) {
  if constexpr (RANK == 3) tma_load_3d(dst, map, 0, 0, row0, bar, policy);
  else tma_load_2d(dst, map, 0, row0, bar, policy);
}

template <bool SWZ>
__device__ __forceinline__ uint32_t tile_off(uint32_t off) {
  if constexpr (SWZ) return swizzle128(off);
  else return off;
}

// One page of a consumer warp: S^T = K_page . Q^T for the group, the online
// softmax update of (m, l) and the rescale of O, then O^T += V_page^T . P^T.
// Ks, Vs: the page's K and V tiles in shared memory; tok0: its first token;
// sc: its (K, V) tile scales (block-scaled pools).
template <int KV, int D, bool PSPLIT>
__device__ __forceinline__ void consume_page(const uint8_t* Ks, const uint8_t* Vs, int tok0, int ctx,
                                             float qk_scale, const uint32_t (&qf)[D / 8],
                                             const uint2* qsm, const float2* sc, float& m0, float& m1,
                                             float& l0, float& l1, float (&o)[D / 16][4], float& vinv) {
  using C = Cfg<KV, D>;
  constexpr bool BF = C::kMmaBf16;
  constexpr bool SWZ = C::kSwizzle;
  constexpr bool F8 = C::kFp8;
  constexpr bool BLK = C::kBlockScaled;
  constexpr int NT = D / 16;
  constexpr bool LDT = F8 && SWZ;
  constexpr bool LD16 = !F8 && SWZ;
  constexpr int KB = D / 4 * C::kElem;  // K bytes per row per thread
  constexpr int VB = D / 8 * C::kElem;  // V bytes per row per thread
  constexpr int RB = C::kRowBytes;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    // ---- issue every shared-memory read of the page up front
    // The page's 16 tokens are taken in a fixed order lambda = 0..15 (the rows
    // of S^T and the K index of P V).  The transposed-ldmatrix path hands each
    // thread tokens 4t .. 4t+3 of a V column, so there lambda = 2t, 2t+1,
    // 2t+8, 2t+9 are the tokens 4t .. 4t+3, and the accumulator rows g, g+8
    // read K rows 2g - (g & 1) and that + 2; otherwise lambda is the token.
    constexpr int VW = VB / 4;  // V words per row per thread
    const int rows[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
    const int kg0 = LDT ? 2 * g - (g & 1) : g, kg1 = LDT ? kg0 + 2 : g + 8;
    uint4 kr[2][KB / 16];
    uint32_t vw[4][VW];
    uint32_t vt[NT][2];  // LDT: V codes, tokens 4t .. 4t+3 of dims 16i + g and 16i + g + 8
    // LD16: V pairs, tokens (2t, 2t+1) of dims 16i + g, 16i + g + 8, then tokens (2t+8, 2t+9)
    uint32_t vh[NT][4];
    {
#pragma unroll
      for (int c = 0; c < KB / 16; ++c) {
        kr[0][c] = lds128(Ks + tile_off<SWZ>(kg0 * RB + t * KB + 16 * c));
        kr[1][c] = lds128(Ks + tile_off<SWZ>(kg1 * RB + t * KB + 16 * c));
      }
      if constexpr (LDT) {
#pragma unroll
        for (int i = 0; i < NT; i += 2)
          ldsm_x2_trans_b8(Vs + tile_off<SWZ>((lane & 15) * RB + 16 * (i + (lane >> 4))), vt[i][0], vt[i][1],
                           vt[i + 1][0], vt[i + 1][1]);
      } else if constexpr (LD16) {
        // matrix m of m-tile i: tokens 8 (m >> 1) .. +7, dims 16i + 8 (m & 1) .. +7
        const uint32_t vrow = ((lane & 7) + ((lane >> 4) << 3)) * RB + ((lane >> 3) & 1) * 16;
#pragma unroll
        for (int i = 0; i < NT; ++i)
          ldsm_x4_trans_b16(Vs + tile_off<SWZ>(vrow + 32 * i), vh[i][0], vh[i][1], vh[i][2], vh[i][3]);
      } else {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t vo = rows[r] * RB + g * VB;
        if constexpr (VB == 8) {
          const uint2 u = lds64(Vs + tile_off<SWZ>(vo));
          vw[r][0] = u.x;
          vw[r][1] = u.y;
        } else {
#pragma unroll
          for (int c = 0; c < VB / 16; ++c) {
            const uint4 u = lds128(Vs + tile_off<SWZ>(vo + 16 * c));
            vw[r][4 * c] = u.x;
            vw[r][4 * c + 1] = u.y;
            vw[r][4 * c + 2] = u.z;
            vw[r][4 * c + 3] = u.w;
          }
        }
      }
      }
    }

    // ---- S^T[token][head] = K_page . Q^T
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < KB / 16; ++c) {
      const uint4 r0 = kr[0][c], r1 = kr[1][c];
      if constexpr (F8) {
        const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w};
        const uint32_t w1[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * c + jj;
          uint32_t af[4];
          e4m3x4_to_f16x2x2(w0[jj], af[0], af[2]);
          e4m3x4_to_f16x2x2(w1[jj], af[1], af[3]);
          const uint2 qj = qsm[j * 32 + lane];
          mma16816<false>(s, af, qj.x, qj.y);
        }
      } else {
        const uint32_t a0[4] = {r0.x, r1.x, r0.y, r1.y};
        mma16816<BF>(s, a0, qf[4 * c], qf[4 * c + 1]);
        const uint32_t a1[4] = {r0.z, r1.z, r0.w, r1.w};
        mma16816<BF>(s, a1, qf[4 * c + 2], qf[4 * c + 3]);
      }
    }

    // ---- online softmax over this page (tokens g and g+8; heads 2t, 2t+1)
    const float qks = BLK ? qk_scale * sc[0].x : qk_scale;
    float x0 = s[0] * qks, x1 = s[1] * qks;
    float x2 = s[2] * qks, x3 = s[3] * qks;
    if (tok0 + 16 > ctx) {  // last, partial page (warp-uniform): slots past ctx hold anything
      if (tok0 + kg0 >= ctx) x0 = x1 = -INFINITY;
      if (tok0 + kg1 >= ctx) x2 = x3 = -INFINITY;
      if constexpr (LDT) {
        const int nv = ctx - tok0 - 4 * t;  // valid tokens among this thread's 4
        const uint32_t keep = nv >= 4 ? 0xFFFFFFFFu : (nv <= 0 ? 0u : (1u << (8 * nv)) - 1u);
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          vt[i][0] &= keep;
          vt[i][1] &= keep;
        }
      } else if constexpr (LD16) {
        const int r0 = ctx - tok0 - 2 * t;  // tokens 2t, 2t+1 valid when r0 > 0, r0 > 1
        const uint32_t klo = (r0 > 0 ? 0x0000FFFFu : 0u) | (r0 > 1 ? 0xFFFF0000u : 0u);
        const uint32_t khi = (r0 > 8 ? 0x0000FFFFu : 0u) | (r0 > 9 ? 0xFFFF0000u : 0u);
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          vh[i][0] &= klo;
          vh[i][1] &= klo;
          vh[i][2] &= khi;
          vh[i][3] &= khi;
        }
      } else {
#pragma unroll
        for (int r = 0; r < 4; ++r)
          if (tok0 + rows[r] >= ctx) {
#pragma unroll
            for (int w = 0; w < VW; ++w) vw[r][w] = 0u;
          }
      }
    }
    float pm0 = fmaxf(x0, x2), pm1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      pm0 = fmaxf(pm0, __shfl_xor_sync(kFull, pm0, off));
      pm1 = fmaxf(pm1, __shfl_xor_sync(kFull, pm1, off));
    }
    // token 0 of every page is valid, so the new maxima are finite
    const float mn0 = fmaxf(m0, pm0), mn1 = fmaxf(m1, pm1);
    // warp-uniform: one scale per page; sv * (1 / vref) > 1 is sv > vref, also
    // for vref = 0 (inf > 1, and 0 * inf is NaN, not > 1)
    const bool vgrow = BLK && sc[0].y * vinv > 1.f;
    if (__any_sync(kFull, (mn0 != m0) | (mn1 != m1)) || vgrow) {  // rescale only when needed
      const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
      l0 *= al0;
      l1 *= al1;
      float ov0 = al0, ov1 = al1;
      if constexpr (BLK) {
        if (vgrow) {
          const float sv = sc[0].y;
          const float r = 1.f / (vinv * sv);  // vref / sv: 0 on the first page with a nonzero scale
          ov0 *= r;
          ov1 *= r;
          vinv = 1.f / sv;
        }
      }
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        o[i][0] *= ov0;
        o[i][1] *= ov1;
        o[i][2] *= ov0;
        o[i][3] *= ov1;
      }
      m0 = mn0;
      m1 = mn1;
    }
    float p0 = fast_exp2(x0 - m0), p1 = fast_exp2(x1 - m1);
    float p2 = fast_exp2(x2 - m0), p3 = fast_exp2(x3 - m1);
    l0 += p0 + p2;
    l1 += p1 + p3;
    if constexpr (BLK) {  // weights of this page's V codes: P * sv / vref
      const float f = sc[0].y * vinv;
      p0 *= f;
      p1 *= f;
      p2 *= f;
      p3 *= f;
    }

    // ---- P^T as the B operand: rows (tokens 2t, 2t+1 | 2t+8, 2t+9), column head g
    const uint32_t plo = pack2<BF>(p0, p1), phi = pack2<BF>(p2, p3);
    const uint32_t pb0 = movmatrix_trans(plo), pb1 = movmatrix_trans(phi);
    uint32_t rb0 = 0, rb1 = 0;
    if constexpr (PSPLIT) {
      const float2 u0 = unpack2<BF>(plo), u1 = unpack2<BF>(phi);
      rb0 = movmatrix_trans(pack2<BF>(p0 - u0.x, p1 - u0.y));
      rb1 = movmatrix_trans(pack2<BF>(p2 - u1.x, p3 - u1.y));
    }

    // ---- O^T[dim][head] += V_page^T . P^T
    {
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        uint32_t af[4];
        if constexpr (LDT) {
          e4m3x4_to_f16x2x2(vt[i][0], af[0], af[2]);
          e4m3x4_to_f16x2x2(vt[i][1], af[1], af[3]);
        } else if constexpr (LD16) {
          af[0] = vh[i][0];
          af[1] = vh[i][1];
          af[2] = vh[i][2];
          af[3] = vh[i][3];
        } else if constexpr (F8) {
          const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
          const uint32_t x01 = __byte_perm(vw[0][i >> 1], vw[1][i >> 1], sel);
          const uint32_t x23 = __byte_perm(vw[2][i >> 1], vw[3][i >> 1], sel);
          e4m3x4_to_f16x2x2(x01, af[0], af[1]);
          e4m3x4_to_f16x2x2(x23, af[2], af[3]);
        } else {
          af[0] = __byte_perm(vw[0][i], vw[1][i], 0x5410u);
          af[1] = __byte_perm(vw[0][i], vw[1][i], 0x7632u);
          af[2] = __byte_perm(vw[2][i], vw[3][i], 0x5410u);
          af[3] = __byte_perm(vw[2][i], vw[3][i], 0x7632u);
        }
        mma16816<BF>(o[i], af, pb0, pb1);
        if constexpr (PSPLIT) mma16816<BF>(o[i], af, rb0, rb1);
      }
    }
}

template <int KV, int D, int OUT, bool PSPLIT, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) decode_kernel(const DecodeArgs a,
                                                          const __grid_constant__ CUtensorMap tmk,
                                                          const __grid_constant__ CUtensorMap tmv) {
  using C = Cfg<KV, D>;
  constexpr bool F8 = C::kFp8;
  constexpr bool BLK = C::kBlockScaled;
  constexpr int NT = D / 16;  // MMA steps along the head dim (QK) / m-tiles (PV)
  // Pools with swizzled rows read V through transposed ldmatrix (the
  // accumulator's dims then follow the ldmatrix layout)
  constexpr bool LDT = F8 && C::kSwizzle;
  constexpr bool LD16 = !F8 && C::kSwizzle;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + C::kAlign - 1) & ~uintptr_t(C::kAlign - 1));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kDataBytes);
  uint64_t* empty = full + C::kStages;
  float2* stage_scale =
      reinterpret_cast<float2*>(smem + C::kDataBytes + 2 * C::kStages * 8 + C::kQBytes);

  // grid (split, kv head, sequence), or (kv head, sequence, split) for the guided layout
  const int split = a.sl.guided ? blockIdx.z : blockIdx.x;
  const int h = a.sl.guided ? blockIdx.x : blockIdx.y;
  const int seq = a.sl.guided ? blockIdx.y : blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();  // the kernel before may still write q, tables, pages

  int ctx = a.ctx[seq];
  if (ctx < 0 || ctx > a.max_blocks * 16) {
    if (threadIdx.x == 0) record_error(a.err, PA_ERR_BOUNDS);
    ctx = ctx < 0 ? 0 : a.max_blocks * 16;
  }
  const int npages = (ctx + 15) >> 4;
  int p_begin, p_end;
  split_pages(a.sl, split, p_begin, p_end);
  const int n_local = max(0, min(npages, p_end) - p_begin);
  // A split past the end of this sequence's pages has nothing to do: no partial
  // is written for it and the merge never reads one.  Split 0 always runs (it
  // writes the zero row of an empty context).
  if (split > 0 && n_local == 0) return;
  // Sequences that fit in one split are finished here, without a merge.
  const bool direct = a.splits == 1 || npages <= first_split_pages(a.sl);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_barrier_init();
  }
  if (threadIdx.x == kConsumerWarps * 32) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  __syncthreads();

  // per-thread softmax state of query heads 2t and 2t+1 (log2 domain)
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const int32_t* trow = a.tables + (size_t)seq * a.max_blocks + p_begin;
    const uint64_t policy = l2_evict_first_policy();
    // Lane i holds the table entry (and, block-scaled, the tile scales) of page
    // base + i.  The next 32 entries are loaded as soon as a batch starts and
    // checked, and their scales fetched, a few pages into it, so no load sits
    // on the path between two batches.
    int issued = 0;
    bool abort = false;
    for (int base = 0; base < n_local && !abort; base += 32) {
      int phys = 0;
      float sk = 0.f, sv = 0.f;
      if (base + lane < n_local) {
        phys = trow[base + lane];
        if (phys < 0 || phys >= a.num_blocks) {
          record_error(a.err, PA_ERR_BOUNDS);
          phys = 0;
        }
        if constexpr (BLK) {
          sk = a.ksc[(size_t)phys * a.Hkv + h];
          sv = a.vsc[(size_t)phys * a.Hkv + h];
        }
      }
      const int cnt = min(32, n_local - base);
      for (int j = 0; j < cnt; ++j) {
        const int ph = __shfl_sync(kFull, phys, j);
        float skj = 0.f, svj = 0.f;
        if constexpr (BLK) {
          skj = __shfl_sync(kFull, sk, j);
          svj = __shfl_sync(kFull, sv, j);
        }
        int stop = 0;
        if (lane == 0) {
          const int k = base + j, stage = k % C::kStages;
          if (k >= C::kStages && !mbar_wait(&empty[stage], ((k / C::kStages) - 1) & 1, pipe_wait_limit())) {
            record_error(a.err, PA_ERR_TIMEOUT);
            stop = 1;
          } else {
            uint8_t* dst = ring + stage * C::kStageBytes;
            const int row0 = (ph * a.Hkv + h) * 16;
            // the scales are published by the same arrive that starts the copies
            if constexpr (BLK) stage_scale[stage] = make_float2(skj, svj);
            mbar_arrive_expect_tx(&full[stage], 2 * C::kTile);
            load_tile<C::kTmaRank>(dst, &tmk, row0, &full[stage], policy);
            load_tile<C::kTmaRank>(dst + C::kTile, &tmv, row0, &full[stage], policy);
            ++issued;
          }
        }
        if (__shfl_sync(kFull, stop, 0)) {
          abort = true;
          break;
        }
      }
    }
    // Wait (bounded) until every copy this CTA issued has landed, so no bulk
    // write can still target the ring when it is reused or the CTA exits.
    if (lane == 0) {
      for (int s = 0; s < C::kStages && s < issued; ++s) {
        const int uses = (issued - 1 - s) / C::kStages + 1;
        if (!mbar_wait(&full[s], (uses - 1) & 1)) record_error(a.err, PA_ERR_TIMEOUT);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    // Q fragment: query head h*G + g (zero when g >= G), dims [t*D/4, (t+1)*D/4)
    constexpr int QW = D / 8;  // 32-bit words per thread
    uint32_t qf[QW];
    float qk_scale = a.qk_scale_log2;
    {
      const uint4* qsrc = reinterpret_cast<const uint4*>(
          a.q + ((size_t)seq * a.Hq + (size_t)h * a.G + g) * D + t * (D / 4));
      uint32_t raw[QW];
#pragma unroll
      for (int c = 0; c < QW / 4; ++c) {
        uint4 u = make_uint4(0, 0, 0, 0);
        if (g < a.G) u = qsrc[c];
        raw[4 * c] = u.x;
        raw[4 * c + 1] = u.y;
        raw[4 * c + 2] = u.z;
        raw[4 * c + 3] = u.w;
      }
      if constexpr (F8) {
        // bfloat16 q -> binary16 with a power-of-two prescale shared by the group
        float amax = 0.f;
#pragma unroll
        for (int w = 0; w < QW; ++w) {
          amax = fmaxf(amax, fabsf(bf16_bits_to_float(raw[w] & 0xFFFFu)));
          amax = fmaxf(amax, fabsf(bf16_bits_to_float(raw[w] >> 16)));
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
        int ex = 0;
        if (amax > 0.f) frexpf(amax, &ex);
        const float qs = amax > 0.f ? ldexpf(1.f, 15 - ex) : 1.f;
        qk_scale = amax > 0.f ? qk_scale * ldexpf(1.f, ex - 15) : qk_scale;
#pragma unroll
        for (int w = 0; w < QW; ++w)
          qf[w] = pack2<false>(bf16_bits_to_float(raw[w] & 0xFFFFu) * qs,
                               bf16_bits_to_float(raw[w] >> 16) * qs);
      } else {
#pragma unroll
        for (int w = 0; w < QW; ++w) qf[w] = raw[w];
      }
    }

    uint2* qsm = nullptr;
    if constexpr (C::kQInSmem) {
      // park the fragments in shared memory: [pair j][lane] (conflict-free 8-byte loads)
      qsm = reinterpret_cast<uint2*>(smem + C::kDataBytes + 2 * C::kStages * 8) + warp * (QW / 2) * 32;
#pragma unroll
      for (int j = 0; j < QW / 2; ++j) qsm[j * 32 + lane] = make_uint2(qf[2 * j], qf[2 * j + 1]);
      __syncwarp();
    }

    // block-scaled pools: V weights are taken relative to the largest V scale
    // this warp has seen (vref), so P * sv / vref stays <= 1 in 16 bits; the
    // accumulator is rescaled when vref grows and multiplied by it at the end
    float vinv = INFINITY;  // 1 / vref; vref starts at 0

    for (int k = warp; k < n_local; k += kConsumerWarps) {
      const int stage = k % C::kStages;
      // every lane waits (acquiring the TMA writes); the outcome is made warp-uniform
      if (!__all_sync(kFull, mbar_wait(&full[stage], (k / C::kStages) & 1, pipe_wait_limit()))) {
        if (lane == 0) record_error(a.err, PA_ERR_TIMEOUT);
        break;
      }
      const uint8_t* Ks = ring + stage * C::kStageBytes;
      const uint8_t* Vs = Ks + C::kTile;
      const int tok0 = (p_begin + k) * 16;
      // (block-scaled pools read the page's (K, V) scales from the stage's slot
      // where they are used: it stays valid until the page is released)

      consume_page<KV, D, PSPLIT>(Ks, Vs, tok0, ctx, qk_scale, qf, qsm, &stage_scale[stage], m0, m1, l0,
                                  l1, o, vinv);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, off);
      l1 += __shfl_xor_sync(kFull, l1, off);
    }
    if constexpr (BLK) {  // back to value units (vref = 0 only if every V here is 0)
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        o[i][0] *= 1.f / vinv;
        o[i][1] *= 1.f / vinv;
        o[i][2] *= 1.f / vinv;
        o[i][3] *= 1.f / vinv;
      }
    }
  }

  grid_dependents_launch();  // the split merge may be scheduled (it waits for this grid)
  __syncthreads();  // the ring is idle from here on: reuse it for the merge

  float* mo = reinterpret_cast<float*>(smem);          // [warp][8 heads][MS]
  constexpr int MS = C::kMergeStride;
  float* mml = mo + kConsumerWarps * 8 * MS;           // [warp][8 heads][2]
  if (warp < kConsumerWarps) {
    const int g = lane >> 2, t = lane & 3;
    float* mw = mo + warp * 8 * MS;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      // output dims held by this thread (accumulator rows g and g + 8 of m-tile i)
      const int d0 = (LDT || LD16) ? 16 * i + g : g * (D / 8) + 2 * i, d1 = (LDT || LD16) ? d0 + 8 : d0 + 1;
      mw[(2 * t) * MS + d0] = o[i][0];
      mw[(2 * t + 1) * MS + d0] = o[i][1];
      mw[(2 * t) * MS + d1] = o[i][2];
      mw[(2 * t + 1) * MS + d1] = o[i][3];
    }
    if (g == 0) {
      float* ml = mml + warp * 16;
      ml[4 * t + 0] = m0;
      ml[4 * t + 1] = l0;
      ml[4 * t + 2] = m1;
      ml[4 * t + 3] = l1;
    }
  }
  __syncthreads();

  const size_t row0 = (size_t)seq * a.Hq + (size_t)h * a.G;
  for (int idx = threadIdx.x; idx < a.G * D; idx += kThreads) {
    const int head = idx / D, dim = idx - head * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mml[w * 16 + 2 * head]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = mml[w * 16 + 2 * head];
        const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
        L += f * mml[w * 16 + 2 * head + 1];
        O += f * mo[(w * 8 + head) * MS + dim];
      }
    }
    if (direct) {
      store_out<OUT>(a.out, (row0 + head) * D + dim, L > 0.f ? O / L * a.v_scale : 0.f);
    } else {
      const size_t prow = (row0 + head) * a.splits + split;
      a.ws_o[prow * D + dim] = O;
      if (dim == 0) {
        a.ws_ml[2 * prow] = M;
        a.ws_ml[2 * prow + 1] = L;
      }
    }
  }
}

// ---------------------------------------------------------------- balanced schedule
// Shared memory of the balanced kernel: the ring and its barriers as in the
// fixed-split kernel, then the per-warp query fragments (FP8 pools), the merge
// slots, the staged query rows of the next unit with its descriptor, and the
// (m, l) exchange of the four warps.
template <int KV, int D>
struct BalCfg {
  using C = Cfg<KV, D>;
  static constexpr int kSlotBytes = 8 * D * 4;      // [8 heads][D] fp32
  // FP8 pools merge through two slots that alias the per-warp query fragments
  // (dead once a unit's last page is done); 16-bit pools keep their fragments
  // in registers and have one slot of their own.
  static constexpr int kMergeSlots = C::kQInSmem ? 2 : 1;
  static_assert(!C::kQInSmem || C::kQBytes == 2 * kSlotBytes, "two merge slots fill the fragment area");
  static constexpr int kOffBars = C::kRingBytes;    // full[S], empty[S], q_full, q_empty
  static constexpr int kOffFrag = kOffBars + (2 * C::kStages + 2) * 8;
  static constexpr int kFragBytes = C::kQInSmem ? C::kQBytes : kSlotBytes;
  static constexpr int kOffQStage = kOffFrag + kFragBytes;  // raw query rows [<= 8][D] (16-bit)
  static constexpr int kOffMl = kOffQStage + 8 * D * 2;     // [4 warps][8 heads] (m, l)
  static constexpr int kOffDesc = kOffMl + kConsumerWarps * 8 * 8;
  // the staged unit's descriptor, then each consumer warp's copy of its current one
  static constexpr int kOffScale = kOffDesc + (1 + kConsumerWarps) * 32;  // block-scaled: [stages] scales
  static constexpr int kSmem = kOffScale + C::kScaleBytes + C::kAlign;
  // The launch asks for at least 48 KiB, so at most four CTAs share an SM
  // (five would need 5 x (48 + 1) KiB, more than the SM's 228 KiB).  The grid
  // is four CTAs per SM with equal page counts; a build that fits five would
  // let the block scheduler put five on some SMs and three on others whenever
  // other work holds part of the GPU as the grid starts (a dependent launch
  // starts before the kernel ahead of it has finished), and the CTAs of a
  // five-CTA SM stream 4/5 as fast, which sets the time of the whole grid.
  static constexpr int kLaunchSmem = kSmem > 48 * 1024 ? kSmem : 48 * 1024;
  // What finishing a unit costs a CTA, in page-times (per-unit traces of a
  // batch of 28-page units: ~3-4 us for the merge, the output rows and the next
  // unit's start, against ~0.3 us a page for FP8 and about twice that for
  // 16-bit pages).
  static constexpr int kUnitCostPages = C::kFp8 ? 12 : 6;
  static_assert(kOffFrag % 16 == 0 && kOffQStage % 16 == 0, "bulk-copy destinations are 16-byte aligned");
};

// The unit the producer hands to the consumers with its query rows.
struct SegDesc {
  int seq, h, pg0, len, ctx, npages, last_cta;
};

// Bounded wait that also gives up once another thread of the CTA has raised
// the abort flag; a wait that runs out raises it and records PA_ERR_TIMEOUT.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (global_ns() - t0 > pipe_wait_limit()) {
      *abort_flag = 1;
      record_error(err, PA_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void consumers_sync() {  // the four consumer warps only
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Balanced schedule.  The grid is one CTA per resident slot.  Every CTA adds
// up the pages of all (sequence, kv head) units from the context lengths on
// the device; the units' pages, in (sequence, kv head, page) order, are cut
// into equal contiguous ranges, one per CTA.  A range crosses unit
// boundaries without draining the pipeline: the producer streams the pages
// of one unit after the other, and ahead of each unit it stages the unit's
// query rows (one bulk copy) and a descriptor; the consumer warps finish a
// unit (merge of their states through shared memory, then the output rows, or
// a partial when the unit goes on in another CTA) while the ring keeps
// filling.  A unit split across CTAs is merged by merge_jobs_kernel: the CTA
// holding its first page records the job.
template <int KV, int D, int OUT, bool PSPLIT, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) decode_bal_kernel(const DecodeArgs a,
                                                              const __grid_constant__ CUtensorMap tmk,
                                                              const __grid_constant__ CUtensorMap tmv) {
  using C = Cfg<KV, D>;
  using B = BalCfg<KV, D>;
  constexpr bool F8 = C::kFp8;
  constexpr bool BLK = C::kBlockScaled;
  constexpr int NT = D / 16;
  constexpr bool LDT = F8 && C::kSwizzle;
  constexpr bool LD16 = !F8 && C::kSwizzle;
  constexpr int QW = D / 8;  // 32-bit query words per thread
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ long long s_warp_sums[kThreads / 32];
  __shared__ long long s_start_off, s_rbegin, s_rend;
  __shared__ int s_start_seq;
  __shared__ int s_abort;
  __shared__ int s_go;
  __shared__ int4 s_job;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + C::kAlign - 1) & ~uintptr_t(C::kAlign - 1));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + B::kOffBars);
  uint64_t* empty = full + C::kStages;
  uint64_t* q_full = empty + C::kStages;
  uint64_t* q_empty = q_full + 1;
  uint8_t* frag = smem + B::kOffFrag;
  const uint16_t* qstage = reinterpret_cast<const uint16_t*>(smem + B::kOffQStage);
  float2* mlx = reinterpret_cast<float2*>(smem + B::kOffMl);  // [warp][head] (m, l)
  SegDesc* desc = reinterpret_cast<SegDesc*>(smem + B::kOffDesc);
  float2* stage_scale = reinterpret_cast<float2*>(smem + B::kOffScale);
  volatile int* abort_flag = &s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();  // the kernel before may still write q, tables, pages

  // ---------------------------------------------------------------- schedule
  // Cost of every sequence (a contiguous share of the sequences per thread)
  // and its prefix sum.  A unit (sequence, kv head) of n pages costs n + kUnit
  // page-times: finishing a unit (the warps' merge, the output rows, the next
  // unit's query rows) costs a CTA about kUnit pages' worth of streaming, so a
  // range of short units gets fewer pages.  Positions: sequence s's units
  // start at the cost of the sequences before s; within a unit the first kUnit
  // positions hold no page, page p sits at kUnit + p.  The ranges are cut in
  // cost; the real pages of position x are R(x) = Hkv * (pages before s) +
  // h * n + max(0, v - kUnit) for x in unit h of s at offset v.
  constexpr int kUnit = B::kUnitCostPages;
  const int per = (a.S + kThreads - 1) / kThreads;
  const int s0 = min(a.S, (int)threadIdx.x * per), s1 = min(a.S, s0 + per);
  long long mine = 0, mine_pg = 0;
  for (int s = s0; s < s1; ++s) {
    int c = a.ctx[s];
    if (c < 0 || c > a.max_blocks * 16) {
      record_error(a.err, PA_ERR_BOUNDS);
      c = clamp_ctx(c, a.max_blocks);
    }
    const int np = (c + 15) >> 4;
    mine_pg += np;
    mine += np > 0 ? (long long)a.Hkv * (np + kUnit) : 0;
  }
  long long total, total_pg;
  const long long before = block_exclusive_scan<kThreads>(mine, s_warp_sums, total);
  __syncthreads();  // the scan's partial sums are read before the second scan writes them
  const long long before_pg = block_exclusive_scan<kThreads>(mine_pg, s_warp_sums, total_pg);
  const long long ptot = total;  // in cost
  const long long T = max((ptot + a.ctas - 1) / a.ctas, (long long)kMinPagesPerCta);
  const long long pos_begin = (long long)blockIdx.x * T;
  const long long pos_end = min(ptot, pos_begin + T);
  // Sequences without context get a zero output row, written by CTA s mod ctas.
  for (int s = blockIdx.x; s < a.S; s += a.ctas) {
    if (a.ctx[s] > 0) continue;
    for (int i = threadIdx.x; i < a.Hq * D; i += kThreads) store_out<OUT>(a.out, (size_t)s * a.Hq * D + i, 0.f);
  }
  // The thread whose sequences hold a boundary finds its sequence and real page.
  auto locate = [&](long long x, bool start) {
    long long cum = before, cum_pg = before_pg * a.Hkv;
    for (int s = s0; s < s1; ++s) {
      const long long np = (clamp_ctx(a.ctx[s], a.max_blocks) + 15) >> 4;
      const long long n = np > 0 ? a.Hkv * (np + kUnit) : 0;
      if (x < cum + n) {
        const long long off = x - cum, hh = off / (np + kUnit), v = off - hh * (np + kUnit);
        const long long r = cum_pg + hh * np + max(0LL, v - kUnit);
        if (start) {
          s_start_seq = s;
          s_start_off = off;
          s_rbegin = r;
        } else {
          s_rend = r;
        }
        return;
      }
      cum += n;
      cum_pg += np * a.Hkv;
    }
  };
  if (before <= pos_begin && pos_begin < before + mine) locate(pos_begin, true);
  if (before <= pos_end && pos_end < before + mine) locate(pos_end, false);
  if (threadIdx.x == 0 && pos_end >= ptot) s_rend = total_pg * a.Hkv;
  if (threadIdx.x == 0 && pos_begin >= ptot) s_rbegin = total_pg * a.Hkv;
  __syncthreads();
  const int n_pages = (int)(s_rend - s_rbegin);  // real pages of this CTA
  if (n_pages <= 0) {  // no pages for this CTA: no partial and no merge job
    if (threadIdx.x == 0) a.jobs[blockIdx.x] = make_int4(-1, 0, 0, 0);
    return;
  }
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_job = make_int4(-1, 0, 0, 0);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, kConsumerWarps);
    fence_barrier_init();
  }
  if (threadIdx.x == kConsumerWarps * 32) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = l2_evict_first_policy();
    int seq = s_start_seq;
    int ctx = clamp_ctx(a.ctx[seq], a.max_blocks);
    int npages = (ctx + 15) >> 4;
    int h = (int)(s_start_off / (npages + kUnit));
    const int v0 = (int)(s_start_off - (long long)h * (npages + kUnit));
    int pg0 = max(0, v0 - kUnit);
    long long ucost = pos_begin - v0;  // cost position of the current unit's start
    int left = n_pages;                // real pages still to stream
    int kb = 0;  // CTA-local index of the unit's first page
    int issued = 0, nq = 0;  // page copies and query-row copies issued (lane 0)
    bool abort = false;
    for (int j = 0; !abort; ++j) {
      const int len = min(npages - pg0, left);
      // the unit's descriptor and query rows, once the consumers hold the previous ones
      int stop = 0;
      if (lane == 0) {
        if (j > 0 && !wait_or_abort(q_empty, (j - 1) & 1, abort_flag, a.err)) {
          stop = 1;
        } else {
          SegDesc sd;
          sd.seq = seq;
          sd.h = h;
          sd.pg0 = pg0;
          sd.len = len;
          sd.ctx = ctx;
          sd.npages = npages;
          sd.last_cta = (int)((ucost + kUnit + npages - 1) / T);  // the CTA of the unit's last page
          *desc = sd;
          const uint32_t qbytes = (uint32_t)(a.G * D * 2);
          mbar_arrive_expect_tx(q_full, qbytes);
          bulk_g2s(smem + B::kOffQStage, a.q + ((size_t)seq * a.Hq + (size_t)h * a.G) * D, qbytes, q_full,
                   policy);
          ++nq;
        }
      }
      if (__shfl_sync(kFull, stop, 0)) break;
      // the unit's pages; lane i holds the table entry (and tile scales) of page base + i
      const int32_t* trow = a.tables + (size_t)seq * a.max_blocks + pg0;
      for (int base = 0; base < len && !abort; base += 32) {
        int phys = 0;
        float sk = 0.f, sv = 0.f;
        if (base + lane < len) {
          phys = trow[base + lane];
          if (phys < 0 || phys >= a.num_blocks) {
            record_error(a.err, PA_ERR_BOUNDS);
            phys = 0;
          }
          if constexpr (BLK) {
            sk = a.ksc[(size_t)phys * a.Hkv + h];
            sv = a.vsc[(size_t)phys * a.Hkv + h];
          }
        }
        const int cnt = min(32, len - base);
        for (int i = 0; i < cnt; ++i) {
          const int ph = __shfl_sync(kFull, phys, i);
          float ski = 0.f, svi = 0.f;
          if constexpr (BLK) {
            ski = __shfl_sync(kFull, sk, i);
            svi = __shfl_sync(kFull, sv, i);
          }
          int st2 = 0;
          if (lane == 0) {
            const int k = kb + base + i, stage = k % C::kStages;
            if (k >= C::kStages && !wait_or_abort(&empty[stage], ((k / C::kStages) - 1) & 1, abort_flag, a.err)) {
              st2 = 1;
            } else {
              uint8_t* dst = ring + stage * C::kStageBytes;
              const int row0 = (ph * a.Hkv + h) * 16;
              if constexpr (BLK) stage_scale[stage] = make_float2(ski, svi);
              mbar_arrive_expect_tx(&full[stage], 2 * C::kTile);
              load_tile<C::kTmaRank>(dst, &tmk, row0, &full[stage], policy);
              load_tile<C::kTmaRank>(dst + C::kTile, &tmv, row0, &full[stage], policy);
              ++issued;
            }
          }
          if (__shfl_sync(kFull, st2, 0)) {
            abort = true;
            break;
          }
        }
      }
      if (abort) break;
      kb += len;
      left -= len;
      if (left <= 0) break;
      // the next unit, from its first page
      ucost += npages + kUnit;
      pg0 = 0;
      if (++h == a.Hkv) {
        h = 0;
        do {  // sequences without pages hold no position; one with pages lies ahead
          if (++seq >= a.S) break;
          ctx = clamp_ctx(a.ctx[seq], a.max_blocks);
        } while (ctx == 0);
        if (seq >= a.S) {  // the lengths changed under the kernel
          if (lane == 0) {
            record_error(a.err, PA_ERR_BOUNDS);
            *abort_flag = 1;
          }
          break;
        }
        npages = (ctx + 15) >> 4;
      }
    }
    // Wait (bounded, whatever the abort flag) until every copy this CTA issued
    // has landed, so no bulk write targets shared memory once the CTA exits.
    if (lane == 0) {
      for (int s = 0; s < C::kStages && s < issued; ++s) {  // each stage's last use
        const int uses = (issued - 1 - s) / C::kStages + 1;
        if (!mbar_wait(&full[s], (uses - 1) & 1)) record_error(a.err, PA_ERR_TIMEOUT);
      }
      if (nq > 0 && !mbar_wait(q_full, (nq - 1) & 1)) record_error(a.err, PA_ERR_TIMEOUT);
    }
    grid_dependents_launch();  // the merge may be scheduled (it waits for this grid)
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3;
    uint32_t qf[QW];
    uint2* qsm = C::kQInSmem ? reinterpret_cast<uint2*>(frag) + warp * (QW / 2) * 32 : nullptr;
    float* slot = reinterpret_cast<float*>(frag);  // merge slot(s) [kMergeSlots][8][D]
    SegDesc* mine_d = desc + 1 + warp;             // this warp's copy of its unit's descriptor
    int kb = 0;
    for (int j = 0; kb < n_pages; ++j) {
      // ---- the unit: descriptor and query rows
      const bool have_q = __all_sync(kFull, wait_or_abort(q_full, j & 1, abort_flag, a.err));
      if (lane == 0) *mine_d = *desc;
      __syncwarp();
      float qk_scale = a.qk_scale_log2;
      {
        uint32_t raw[QW];
        const uint4* qrow = reinterpret_cast<const uint4*>(qstage + g * D + t * (D / 4));
#pragma unroll
        for (int c = 0; c < QW / 4; ++c) {
          uint4 u = make_uint4(0, 0, 0, 0);
          if (g < a.G && have_q) u = qrow[c];
          raw[4 * c] = u.x;
          raw[4 * c + 1] = u.y;
          raw[4 * c + 2] = u.z;
          raw[4 * c + 3] = u.w;
        }
        if constexpr (F8) {
          // bfloat16 q -> binary16 with a power-of-two prescale shared by the group
          float amax = 0.f;
#pragma unroll
          for (int w = 0; w < QW; ++w) {
            amax = fmaxf(amax, fabsf(bf16_bits_to_float(raw[w] & 0xFFFFu)));
            amax = fmaxf(amax, fabsf(bf16_bits_to_float(raw[w] >> 16)));
          }
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
          int ex = 0;
          if (amax > 0.f) frexpf(amax, &ex);
          const float qs = amax > 0.f ? ldexpf(1.f, 15 - ex) : 1.f;
          qk_scale = amax > 0.f ? qk_scale * ldexpf(1.f, ex - 15) : qk_scale;
#pragma unroll
          for (int w = 0; w < QW; ++w)
            qf[w] = pack2<false>(bf16_bits_to_float(raw[w] & 0xFFFFu) * qs,
                                 bf16_bits_to_float(raw[w] >> 16) * qs);
        } else {
#pragma unroll
          for (int w = 0; w < QW; ++w) qf[w] = raw[w];
        }
      }
      if constexpr (C::kQInSmem) {
#pragma unroll
        for (int i = 0; i < QW / 2; ++i) qsm[i * 32 + lane] = make_uint2(qf[2 * i], qf[2 * i + 1]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(q_empty);  // the staged rows and descriptor may be replaced

      // ---- the unit's pages: warp w takes those whose CTA-local index is w mod 4
      const int len = have_q ? mine_d->len : 0;
      const int pg0 = mine_d->pg0, ctx = mine_d->ctx;
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      float o[NT][4];
#pragma unroll
      for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      float vinv = INFINITY;  // block-scaled pools: 1 / the largest V scale seen (see decode_kernel)
      for (int k = kb + ((warp - kb) & (kConsumerWarps - 1)); k < kb + len; k += kConsumerWarps) {
        const int stage = k % C::kStages;
        if (!__all_sync(kFull, wait_or_abort(&full[stage], (k / C::kStages) & 1, abort_flag, a.err))) break;
        const uint8_t* Ks = ring + stage * C::kStageBytes;
        consume_page<KV, D, PSPLIT>(Ks, Ks + C::kTile, (pg0 + k - kb) * 16, ctx, qk_scale, qf, qsm,
                                    &stage_scale[stage], m0, m1, l0, l1, o, vinv);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(kFull, l0, off);
        l1 += __shfl_xor_sync(kFull, l1, off);
      }
      if constexpr (BLK) {  // back to value units
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          o[i][0] *= 1.f / vinv;
          o[i][1] *= 1.f / vinv;
          o[i][2] *= 1.f / vinv;
          o[i][3] *= 1.f / vinv;
        }
      }

      // ---- merge of the four warps' states for this unit
      if (g == 0) {
        mlx[warp * 8 + 2 * t] = make_float2(m0, l0);
        mlx[warp * 8 + 2 * t + 1] = make_float2(m1, l1);
      }
      consumers_sync();  // every warp is past its last page (fragments dead); (m, l) published
      float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        M0 = fmaxf(M0, mlx[w * 8 + 2 * t].x);
        M1 = fmaxf(M1, mlx[w * 8 + 2 * t + 1].x);
      }
      const float f0 = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - M0);
      const float f1 = (m1 == -INFINITY) ? 0.f : fast_exp2(m1 - M1);
      // A slot holds the accumulator fragments as the lanes hold them: value c
      // of m-tile i of lane L at (i * 4 + c) * 32 + L (stores without bank conflicts)
#pragma unroll
      for (int step = 0; step < kConsumerWarps / B::kMergeSlots; ++step) {
        if (warp / B::kMergeSlots == step) {
          float* sl = slot + (warp % B::kMergeSlots) * 8 * D + lane;
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            const float v[4] = {o[i][0] * f0, o[i][1] * f1, o[i][2] * f0, o[i][3] * f1};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              if (step == 0) sl[(i * 4 + c) * 32] = v[c];
              else sl[(i * 4 + c) * 32] += v[c];
            }
          }
        }
        consumers_sync();
      }
      // ---- the unit's output rows, or its partial
      const SegDesc sd = *mine_d;
      const bool direct = sd.pg0 == 0 && sd.len == sd.npages;
      const int pslot = 2 * blockIdx.x + (j == 0 ? 0 : 1);
      const bool write = have_q && !*abort_flag;
      if (write && !direct && sd.pg0 == 0 && threadIdx.x == 0) s_job = make_int4(sd.seq, sd.h, sd.last_cta, pslot);
      const int tid = threadIdx.x;  // 0 .. 127
      for (int idx = tid; idx < a.G * D && write; idx += kConsumerWarps * 32) {
        const int head = idx / D, dim = idx - head * D;
        // where the fragments hold (head, dim): rows g (+ 8) of m-tile i for the
        // transposed-ldmatrix layouts, columns 2i (+ 1) of row g otherwise
        int i, gg, hi;
        if constexpr (LDT || LD16) {
          i = dim >> 4;
          gg = dim & 7;
          hi = (dim >> 3) & 1;
        } else {
          gg = dim / (D / 8);
          i = (dim % (D / 8)) >> 1;
          hi = dim & 1;
        }
        const int sidx = (i * 4 + 2 * hi + (head & 1)) * 32 + 4 * gg + (head >> 1);
        float O = slot[sidx];
        if constexpr (B::kMergeSlots == 2) O += slot[8 * D + sidx];
        float M = -INFINITY, L = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mlx[w * 8 + head].x);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float2 ml = mlx[w * 8 + head];
          L += (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M) * ml.y;
        }
        if (direct) {
          const size_t row = (size_t)sd.seq * a.Hq + (size_t)sd.h * a.G + head;
          store_out<OUT>(a.out, row * D + dim, L > 0.f ? O / L * a.v_scale : 0.f);
        } else {
          const size_t prow = (size_t)pslot * a.G + head;
          a.ws_o[prow * D + dim] = O;
          if (dim == 0) {
            a.ws_ml[2 * prow] = M;
            a.ws_ml[2 * prow + 1] = L;
          }
        }
      }
      if (tid == 0) s_go = !*abort_flag;  // one thread decides for all, read after the barrier
      consumers_sync();  // the slots and the (m, l) area are free again
      kb += len;
      if (!s_go) break;  // uniform: every warp reads the one decision
    }
    grid_dependents_launch();
    if (threadIdx.x == 0) a.jobs[blockIdx.x] = s_job;
  }
}

// Merge of the per-split partial states, M = max m_i, L = sum l_i 2^(m_i - M),
// O = sum o_i 2^(m_i - M) / L, over the splits the sequence used (rows of
// sequences that fit one split were written by the decode kernel itself).
__device__ __forceinline__ int used_splits(const int32_t* ctx, int seq, int max_blocks, const SplitLayout& L) {
  int c = ctx[seq];
  c = c < 0 ? 0 : min(c, max_blocks * 16);
  const int np = (c + 15) / 16;
  if (!L.guided) return (np + L.pps - 1) / L.pps;
  int n = 0;
#pragma unroll
  for (int i = 0; i < kGuidedSplits; ++i) n += (i < L.splits && L.b[i] < np) ? 1 : 0;
  return n;
}

// Few splits (at most 8): one warp per (sequence, query head).  Lane s reads
// split s's (m, l), so M and L are one load and a warp reduction away; the
// lanes then read every split's slice of O (D / 32 values each) at once, and
// add them up in split order.
template <int D, int OUT>
__global__ void __launch_bounds__(128) reduce_rows_kernel(const float* __restrict__ ws_o,
                                                          const float* __restrict__ ws_ml,
                                                          const int32_t* __restrict__ ctx,
                                                          void* out, int rows, int Hq, int splits,
                                                          int max_blocks, const SplitLayout sl, float v_scale) {
  grid_dependency_wait();  // the partials come from the decode kernel just before
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int n = min(splits, used_splits(ctx, row / Hq, max_blocks, sl));
  if (n <= 1) return;
  constexpr int PER = D / 32;
  float ms = -INFINITY, ls = 0.f;
  if (lane < n) {
    const float2 v = reinterpret_cast<const float2*>(ws_ml)[(size_t)row * splits + lane];
    ms = v.x;
    ls = v.y;
  }
  float M = ms;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
  const float w = (ms == -INFINITY) ? 0.f : fast_exp2(ms - M);  // 0 for lanes >= n
  float L = w * ls;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
  float O[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) O[j] = 0.f;
  const float* po = ws_o + (size_t)row * splits * D + lane * PER;
  float v[8][PER];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    if (s < n) {
      if constexpr (PER == 4) {
        const float4 x = *reinterpret_cast<const float4*>(po + (size_t)s * D);
        v[s][0] = x.x;
        v[s][1] = x.y;
        v[s][2] = x.z;
        v[s][3] = x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(po + (size_t)s * D);
        v[s][0] = x.x;
        v[s][1] = x.y;
      }
    }
  }
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const float f = __shfl_sync(kFull, w, s);
    if (s < n) {
#pragma unroll
      for (int j = 0; j < PER; ++j) O[j] += f * v[s][j];
    }
  }
  const float inv = L > 0.f ? v_scale / L : 0.f;
#pragma unroll
  for (int j = 0; j < PER; ++j) store_out<OUT>(out, (size_t)row * D + lane * PER + j, O[j] * inv);
}

// Many splits: one 128-thread CTA per row; the split weights are computed
// once into shared memory and every thread (one head dim each) streams its
// column of partials with independent loads.
template <int D, int OUT>
__global__ void __launch_bounds__(128) reduce_wide_kernel(const float* __restrict__ ws_o,
                                                          const float* __restrict__ ws_ml,
                                                          const int32_t* __restrict__ ctx,
                                                          void* out, int Hq, int splits,
                                                          int max_blocks, const SplitLayout sl, float v_scale) {
  grid_dependency_wait();
  __shared__ float wsh[128];
  __shared__ float red[4];
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = min(splits, used_splits(ctx, row / Hq, max_blocks, sl));
  if (n <= 1) return;
  const float* ml = ws_ml + (size_t)row * splits * 2;
  float m = -INFINITY;
  for (int s = tid; s < n; s += 128) m = fmaxf(m, ml[2 * s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  float L = 0.f, O = 0.f;
  for (int base = 0; base < n; base += 128) {
    const int s = base + tid;
    float w = 0.f;
    if (s < n && M != -INFINITY) {
      const float ms = ml[2 * s];
      w = (ms == -INFINITY) ? 0.f : fast_exp2(ms - M);
      L += w * ml[2 * s + 1];
    }
    wsh[tid] = w;
    __syncthreads();
    const int cnt = min(128, n - base);
    if (tid < D) {
      // 16 independent loads per round into four partial sums: the merge is
      // bound by load latency, not bandwidth
      const float* po = ws_o + ((size_t)row * splits + base) * D + tid;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      int j = 0;
      for (; j + 16 <= cnt; j += 16) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = po[(size_t)(j + e) * D];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e & 3] += wsh[j + e] * v[e];
      }
      for (; j < cnt; ++j) acc[0] += wsh[j] * po[(size_t)j * D];
      O += (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
  if (lane == 0) red[warp] = L;
  __syncthreads();
  L = red[0] + red[1] + red[2] + red[3];
  if (tid < D) store_out<OUT>(out, (size_t)row * D + tid, L > 0.f ? O * (v_scale / L) : 0.f);
}

// Balanced schedule: the merge of each unit whose pages span several CTAs.
// CTA (c, head) takes CTA c's job, if any: the unit whose first page CTA c
// holds and which goes on past c's range.  Its pieces are CTA c's partial (in
// slot job.w) and the first-segment partials (slot 2c') of CTAs c' = c + 1 ..
// job.z, in that order; M = max m_i, L = sum l_i 2^(m_i - M),
// O = sum o_i 2^(m_i - M) / L.  Whole units were written by the decode kernel.
template <int D, int OUT>
__global__ void __launch_bounds__(128) merge_jobs_kernel(const float* __restrict__ ws_o,
                                                         const float* __restrict__ ws_ml,
                                                         const int4* __restrict__ jobs, void* out,
                                                         int Hq, int G, float v_scale) {
  grid_dependency_wait();  // the partials and jobs come from the decode kernel just before
  __shared__ float wsh[128];
  __shared__ float red[4];
  const int c0 = blockIdx.x, head = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int4 job = jobs[c0];
  if (job.x < 0) return;
  const int n = job.z - c0 + 1;  // pieces
  // partial row of piece i: slot job.w for i = 0, else 2 (c0 + i)
#define PA_PROW(i) ((size_t)((i) == 0 ? job.w : 2 * (c0 + (i))) * G + head)
  float m = -INFINITY;
  for (int i = tid; i < n; i += 128) m = fmaxf(m, ws_ml[2 * PA_PROW(i)]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  float L = 0.f, O = 0.f;
  for (int base = 0; base < n; base += 128) {
    const int i = base + tid;
    float w = 0.f;
    if (i < n && M != -INFINITY) {
      const float mi = ws_ml[2 * PA_PROW(i)];
      w = (mi == -INFINITY) ? 0.f : fast_exp2(mi - M);
      L += w * ws_ml[2 * PA_PROW(i) + 1];
    }
    wsh[tid] = w;
    __syncthreads();
    const int cnt = min(128, n - base);
    if (tid < D) {
      // 16 independent loads per round into four partial sums (latency-bound)
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      int j = 0;
      for (; j + 16 <= cnt; j += 16) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = ws_o[PA_PROW(base + j + e) * D + tid];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e & 3] += wsh[j + e] * v[e];
      }
      for (; j < cnt; ++j) acc[0] += wsh[j] * ws_o[PA_PROW(base + j) * D + tid];
      O += (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
    __syncthreads();
  }
#undef PA_PROW
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
  if (lane == 0) red[warp] = L;
  __syncthreads();
  L = red[0] + red[1] + red[2] + red[3];
  const size_t row = (size_t)job.x * Hq + (size_t)job.y * G + head;
  if (tid < D) store_out<OUT>(out, row * D + tid, L > 0.f ? O * (v_scale / L) : 0.f);
}

// ---------------------------------------------------------------- host side
struct KernelInfo {
  const void* fn;
  int smem;
  int occupancy[128];  // per device, 0 = not yet configured
};

template <int KV, int D, int OUT>
struct Launcher {
  static constexpr bool kPsplit = (KV == KV_BF16) || (OUT == OUT_F32);
  static constexpr int kMinB = Cfg<KV, D>::kMinBlocks, kMinBLow = Cfg<KV, D>::kMinBlocksLow;
  static KernelInfo& info() {
    static KernelInfo ki = {reinterpret_cast<const void*>(&decode_kernel<KV, D, OUT, kPsplit, kMinB>),
                            Cfg<KV, D>::kSmem,
                            {}};
    return ki;
  }
  // the build for launches with at most kMinBLow CTAs per SM (the same kernel
  // unless the pool type has a second build)
  static KernelInfo& info_low() {
    if constexpr (kMinBLow == kMinB) {
      return info();
    } else {
      static KernelInfo ki = {reinterpret_cast<const void*>(&decode_kernel<KV, D, OUT, kPsplit, kMinBLow>),
                              Cfg<KV, D>::kSmem,
                              {}};
      return ki;
    }
  }
  // the balanced-schedule build
  static KernelInfo& info_bal() {
    static KernelInfo ki = {reinterpret_cast<const void*>(&decode_bal_kernel<KV, D, OUT, kPsplit, kMinB>),
                            BalCfg<KV, D>::kLaunchSmem,
                            {}};
    return ki;
  }
  // Both kernels are launched with programmatic stream serialization: each may
  // be scheduled while the kernel before it in the stream finishes, and waits
  // for it before its first global access, so its launch overlaps that
  // kernel's tail (decode + merge of a 4 x 131072 batch 1.2% faster, behind
  // its cache write; 0.6% with the merge alone launched so).
  static cudaError_t launch(const DecodeArgs& a, const CUtensorMap* tk, const CUtensorMap* tv,
                            int S, cudaStream_t st, bool low, bool bal) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<KV, D>::kSmem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (bal) {
      cfg.gridDim = dim3(a.ctas);
      cfg.dynamicSmemBytes = BalCfg<KV, D>::kLaunchSmem;
      cudaError_t e = cudaLaunchKernelEx(&cfg, decode_bal_kernel<KV, D, OUT, kPsplit, kMinB>, a, *tk, *tv);
      if (e != cudaSuccess) return e;
      cfg.gridDim = dim3(a.ctas, a.G);
      cfg.blockDim = dim3(128);
      cfg.dynamicSmemBytes = 0;
      return cudaLaunchKernelEx(&cfg, merge_jobs_kernel<D, OUT>, (const float*)a.ws_o, (const float*)a.ws_ml,
                                (const int4*)a.jobs, a.out, a.Hq, a.G, a.v_scale);
    }
    cfg.gridDim = a.sl.guided ? dim3(a.Hkv, S, a.splits) : dim3(a.splits, a.Hkv, S);
    cudaError_t e = low ? cudaLaunchKernelEx(&cfg, decode_kernel<KV, D, OUT, kPsplit, kMinBLow>, a, *tk, *tv)
                        : cudaLaunchKernelEx(&cfg, decode_kernel<KV, D, OUT, kPsplit, kMinB>, a, *tk, *tv);
    if (e != cudaSuccess || a.splits == 1) return e;
    const int rows = S * a.Hq;
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    if (a.splits <= 8) {
      cfg.gridDim = dim3((rows + 3) / 4);
      e = cudaLaunchKernelEx(&cfg, reduce_rows_kernel<D, OUT>, (const float*)a.ws_o, (const float*)a.ws_ml,
                             a.ctx, a.out, rows, a.Hq, a.splits, a.max_blocks, a.sl, a.v_scale);
    } else {
      cfg.gridDim = dim3(rows);
      e = cudaLaunchKernelEx(&cfg, reduce_wide_kernel<D, OUT>, (const float*)a.ws_o, (const float*)a.ws_ml,
                             a.ctx, a.out, a.Hq, a.splits, a.max_blocks, a.sl, a.v_scale);
    }
    return e;
  }
};

struct Dispatch {
  KernelInfo* info;      // the default build (its occupancy sizes the splits)
  KernelInfo* info_low;  // the build for launches of one wave at its own occupancy
  KernelInfo* info_bal;  // the balanced-schedule build
  cudaError_t (*launch)(const DecodeArgs&, const CUtensorMap*, const CUtensorMap*, int,
                        cudaStream_t, bool, bool);
};

// ---- TMA descriptors of the pool regions
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A map over one layer's K (or V) region seen as rows of one token of one kv
// head (row_bytes = head_dim * elem_bytes); a box is one 16-row tile.  Rows of
// 256 bytes are described as [rows][2][128] so every box row is 128 bytes, the
// largest the 128-byte swizzle accepts.
int make_tile_map(CUtensorMap* m, void* base, int row_bytes, long long rows) {
  EncodeTiledFn f = encode_tiled();
  if (!f) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const CUtensorMapSwizzle swz =
      (row_bytes % 128 == 0) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r;
  if (row_bytes == 256) {
    const cuuint64_t dims[3] = {128, 2, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {128, 256};
    const cuuint32_t box[3] = {128, 2, 16};
    const cuuint32_t es[3] = {1, 1, 1};
    r = f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)row_bytes, 16};
    const cuuint32_t es[2] = {1, 1};
    r = f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PA_OK;
}

// The K and V maps of `layer`, encoded on first use (shared with the prefill).
int layer_maps(pa_pool* pool, int layer, const CUtensorMap** tk, const CUtensorMap** tv) {
  static_assert(sizeof(CUtensorMap) == sizeof(pa_tmap_blob), "tensor map size");
  const pa_pool_desc& d = pool->desc;
  if (pool->tmaps.size() != 2u * d.n_layers) {
    pool->tmaps.assign(2u * d.n_layers, pa_tmap_blob{});
    pool->tmap_ready.assign(d.n_layers, 0);
  }
  CUtensorMap* maps = reinterpret_cast<CUtensorMap*>(pool->tmaps.data());
  if (!pool->tmap_ready[layer]) {
    const int row_bytes = d.head_dim * pool->elem_bytes;
    const long long rows = (long long)d.num_blocks * d.n_kv_heads * d.block_size;
    int st = make_tile_map(&maps[2 * layer], pool->k + (size_t)layer * pool->layer_bytes,
                           row_bytes, rows);
    if (st) return st;
    st = make_tile_map(&maps[2 * layer + 1], pool->v + (size_t)layer * pool->layer_bytes,
                       row_bytes, rows);
    if (st) return st;
    pool->tmap_ready[layer] = 1;
  }
  *tk = &maps[2 * layer];
  *tv = &maps[2 * layer + 1];
  return PA_OK;
}

int layer_half_maps(pa_pool* pool, int layer, const CUtensorMap** tk, const CUtensorMap** tv) {
  const pa_pool_desc& d = pool->desc;
  const int row_bytes = d.head_dim * pool->elem_bytes;
  if (row_bytes != 256) return fail(PA_ERR_UNSUPPORTED, "half-row maps need 256-byte rows");
  if (pool->tmaps_half.size() != 2u * d.n_layers) {
    pool->tmaps_half.assign(2u * d.n_layers, pa_tmap_blob{});
    pool->tmap_half_ready.assign(d.n_layers, 0);
  }
  CUtensorMap* maps = reinterpret_cast<CUtensorMap*>(pool->tmaps_half.data());
  if (!pool->tmap_half_ready[layer]) {
    EncodeTiledFn f = encode_tiled();
    if (!f) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t rows = (cuuint64_t)d.num_blocks * d.n_kv_heads * d.block_size;
    const cuuint64_t dims[2] = {256, rows};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {128, 16};
    const cuuint32_t es[2] = {1, 1};
    for (int which = 0; which < 2; ++which) {
      uint8_t* base = (which ? pool->v : pool->k) + (size_t)layer * pool->layer_bytes;
      CUresult r = f(&maps[2 * layer + which], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
    pool->tmap_half_ready[layer] = 1;
  }
  *tk = &maps[2 * layer];
  *tv = &maps[2 * layer + 1];
  return PA_OK;
}

template <int KV, int D, int OUT>
Dispatch make_dispatch() {
  return {&Launcher<KV, D, OUT>::info(), &Launcher<KV, D, OUT>::info_low(), &Launcher<KV, D, OUT>::info_bal(),
          &Launcher<KV, D, OUT>::launch};
}

template <int KV, int D>
Dispatch pick_out(int out_dtype) {
  if (out_dtype == PA_FP32) return make_dispatch<KV, D, OUT_F32>();
  if constexpr (KV == KV_F16) return make_dispatch<KV, D, OUT_F16>();
  else return make_dispatch<KV, D, OUT_BF16>();
}

template <int KV>
Dispatch pick_d(int head_dim, int out_dtype) {
  return head_dim == 64 ? pick_out<KV, 64>(out_dtype) : pick_out<KV, 128>(out_dtype);
}

Dispatch pick(int kv_dtype, int head_dim, int out_dtype) {
  switch (kv_dtype) {
    case PA_FP16:
      return pick_d<KV_F16>(head_dim, out_dtype);
    case PA_BF16:
      return pick_d<KV_BF16>(head_dim, out_dtype);
    case PA_FP8_E4M3_BLOCK:
      return pick_d<KV_E4M3B>(head_dim, out_dtype);
    default:
      return pick_d<KV_E4M3>(head_dim, out_dtype);
  }
}

// Sets the shared-memory opt-in once per device and returns resident CTAs per SM.
int configure(KernelInfo& ki, int dev) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 128) return 0;
  if (ki.occupancy[dev] > 0) return ki.occupancy[dev];
  if (cudaFuncSetAttribute(ki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem) !=
      cudaSuccess)
    return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, ki.fn, kThreads, ki.smem) != cudaSuccess)
    return 0;
  ki.occupancy[dev] = occ > 0 ? occ : 1;
  return ki.occupancy[dev];
}

int in_dtype_of(int kv_dtype) { return kv_dtype == PA_FP16 ? PA_FP16 : PA_BF16; }

int check_shape(const pa_pool* pool, int S, int n_q_heads, int max_blocks) {
  if (!pool) return fail(PA_ERR_INVALID, "null pool");
  if (S < 0 || max_blocks < 1 || n_q_heads < 1)
    return fail(PA_ERR_INVALID, "need S >= 0, max_blocks_per_seq >= 1, n_q_heads >= 1");
  const int hkv = pool->desc.n_kv_heads;
  if (n_q_heads % hkv != 0)
    return fail(PA_ERR_INVALID, "n_q_heads %d is not a multiple of n_kv_heads %d", n_q_heads, hkv);
  if (n_q_heads / hkv > 8)
    return fail(PA_ERR_UNSUPPORTED, "query heads per kv head must be <= 8 (got %d)",
                n_q_heads / hkv);
  if (S > 65535) return fail(PA_ERR_UNSUPPORTED, "at most 65535 sequences per call");
  if (hkv > 65535) return fail(PA_ERR_UNSUPPORTED, "at most 65535 kv heads");
  return PA_OK;
}

// Splits along the pages.  With u = S * Hkv units of at most B pages, s splits
// give u * s CTAs of P = ceil(B / s) pages, launched in waves of r = occ * sms
// resident CTAs.  Once an SM holds about k_sat CTAs the kernel is bound by its
// share of HBM bandwidth, so a wave whose busiest SM holds k CTAs lasts about
// (P + c) * max(k, k_sat) page-times: k CTAs share the SM's bandwidth, and fewer
// than k_sat cannot fill it (each is then bound by its own load latency).  The
// cost of s is the sum over its waves; c is the fixed cost of a CTA (pipeline
// fill, query load) plus, with splits, its partial and merge.  Measured on the
// 70B-shaped FP8 batches this ranks the split counts as the kernel does (4 x
// 131072 tokens: 19 splits, exactly 4 CTAs per SM, best; 256 x 4096: 1 split).
// The contexts live on the device, so every unit is taken as full: a batch with
// a few sequences much longer than the rest is better served by an explicit
// split count.
// SMs of the current device and resident CTAs per SM of the decode kernel's
// default build for this pool (the query dtype's output).
int decode_residency(const pa_pool* pool, int* sms, int* occ) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
  Dispatch d = pick(pool->desc.kv_dtype, pool->desc.head_dim, in_dtype_of(pool->desc.kv_dtype));
  *occ = configure(*d.info, dev);
  if (*occ <= 0) return fail(PA_ERR_CUDA, "decode kernel occupancy query failed");
  return PA_OK;
}

int auto_splits(const pa_pool* pool, int S, int max_blocks, int* out) {
  int sms = 0, occ = 0;
  int st = decode_residency(pool, &sms, &occ);
  if (st) return st;
  const double slots = (double)sms * occ;
  const double k_sat = std::min(4, occ);
  const double units = (double)std::max(S, 1) * pool->desc.n_kv_heads;
  const int max_s = std::min(max_blocks, 256);
  int best = 1;
  double best_cost = 1e300;
  for (int s = 1; s <= max_s; ++s) {
    const int pps = (max_blocks + s - 1) / s;
    if (s > 1 && (max_blocks + pps - 1) / pps != s) continue;  // same as a smaller s
    const double ctas = units * s;
    const double full_waves = std::floor(ctas / slots);
    const double rest = ctas - full_waves * slots;
    double per_sm = full_waves * std::max((double)occ, k_sat);
    if (rest > 0) per_sm += std::max(std::ceil(rest / sms), k_sat);
    const double cost = per_sm * (pps + 4.0 + (s > 1 ? 2.0 : 0.0));
    if (cost < best_cost * 0.97) {  // more splits only for a clear gain
      best_cost = cost;
      best = s;
    }
  }
  *out = best;
  return PA_OK;
}

// Guided layout over `max_blocks` table columns in `want` <= kGuidedSplits
// splits: split k's share of the columns is proportional to kGuidedRatio^k
// (fewer splits when the table is too narrow for all of them to hold a
// column).  Returns the split count n; b[0] = 0 < b[1] < ... < b[n] = max_blocks.
// The ratio: on the 8B-shaped ragged FP8 batch (64 sequences of 512 to 4096
// tokens, two and a half waves of CTAs) 0.55 measured best among 0.5 .. 0.65.
constexpr double kGuidedRatio = 0.55;
int guided_bounds(int max_blocks, int want, int* b) {
  double w[kGuidedSplits], sum = 0.0;
  for (int k = 0; k < want; ++k) sum += (w[k] = std::pow(kGuidedRatio, k));
  int n = 0;
  b[0] = 0;
  double cum = 0.0;
  for (int k = 0; k < want; ++k) {
    cum += w[k];
    const int e = k == want - 1 ? max_blocks : (int)std::lround(cum / sum * max_blocks);
    if (e > b[n]) b[++n] = e;
  }
  return n;
}

int resolve_splits(const pa_pool* pool, int S, int max_blocks, int num_splits, int* splits,
                   int* pps) {
  int s = num_splits;
  if (s < 0) return fail(PA_ERR_INVALID, "num_splits must be >= 0");
  if (s == 0) {
    int st = auto_splits(pool, S, max_blocks, &s);
    if (st) return st;
  }
  s = std::max(1, std::min(s, max_blocks));
  if (s > 65535) s = 65535;
  const int p = (max_blocks + s - 1) / s;
  *pps = p;
  *splits = (max_blocks + p - 1) / p;
  return PA_OK;
}

// The balanced schedule takes batches of up to this many sequences (every CTA
// scans the context lengths, so the scan must stay short).
constexpr int kBalancedMaxSeqs = 4096;

// How one pa_decode call runs: fixed splits (grid (splits, kv head, sequence))
// or the balanced schedule (one CTA per resident slot), and its workspace.
struct Plan {
  bool bal = false;
  int splits = 1, pps = 1;  // fixed splits
  bool guided = false;      // fixed splits in the guided layout, bounds b
  int b[kGuidedSplits + 1] = {};
  int ctas = 0;             // balanced schedule
  size_t ws_bytes = 0;
};

size_t fixed_ws_bytes(int S, int n_q_heads, int splits, int head_dim) {
  return splits > 1 ? (size_t)S * n_q_heads * splits * (head_dim + 2) * sizeof(float) : 0;
}

// per CTA: two partial slots of G rows of (D + 2) floats, and one 16-byte job
size_t bal_ws_per_cta(int G, int head_dim) { return 2 * (size_t)G * (head_dim + 2) * sizeof(float) + 16; }

// num_splits = PA_SPLITS_BALANCED: the balanced schedule with one CTA per
// resident slot of its build, at most four per SM (the occupancy of the query
// dtype's build, so the workspace size does not depend on the output dtype).
// Otherwise fixed splits (num_splits, or the wave model's count for 0).  cap >
// 0 bounds the workspace (the no-allocation entry point): the balanced
// schedule then uses at most cap / bal_ws_per_cta CTAs, an automatic split
// count is lowered until its partials fit, and an explicit count whose
// partials do not fit is rejected.
int make_plan(const pa_pool* pool, int S, int n_q_heads, int max_blocks, int num_splits,
              size_t cap, Plan* p) {
  *p = Plan();
  if (num_splits < 0 && num_splits != PA_SPLITS_BALANCED)
    return fail(PA_ERR_INVALID, "num_splits must be >= 0 or PA_SPLITS_BALANCED");
  const int G = n_q_heads / pool->desc.n_kv_heads, D = pool->desc.head_dim;
  if (num_splits == PA_SPLITS_BALANCED) {
    if (S > kBalancedMaxSeqs)
      return fail(PA_ERR_UNSUPPORTED, "the balanced schedule takes at most %d sequences (got %d)",
                  kBalancedMaxSeqs, S);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
    Dispatch d = pick(pool->desc.kv_dtype, D, in_dtype_of(pool->desc.kv_dtype));
    const int occ = configure(*d.info_bal, dev);
    if (occ <= 0) return fail(PA_ERR_CUDA, "decode kernel occupancy query failed");
    // at most four CTAs per SM: with long units four stream as fast as five
    // and each has a quarter more of the SM's bandwidth
    long long ctas = (long long)std::min(occ, 4) * sms;
    if (cap > 0) ctas = std::min<long long>(ctas, (long long)(cap / bal_ws_per_cta(G, D)));
    if (ctas < 1) return fail(PA_ERR_INVALID, "the balanced schedule's partials do not fit the scratch");
    p->bal = true;
    p->ctas = (int)ctas;
    p->splits = 0;
    p->ws_bytes = (size_t)ctas * bal_ws_per_cta(G, D);
    return PA_OK;
  }
  int st = resolve_splits(pool, S, max_blocks, num_splits, &p->splits, &p->pps);
  if (st) return st;
  const size_t row_bytes = (size_t)S * n_q_heads * (D + 2) * sizeof(float);
  if (cap > 0 && p->splits > 1 && row_bytes * p->splits > cap) {
    if (num_splits != 0)
      return fail(PA_ERR_INVALID,
                  "pa_decode_no_alloc: %d splits (num_splits %d resolved against %d table "
                  "columns) need %zu bytes of scratch, above the static maximum of %zu bytes "
                  "(use fewer splits, or pa_decode with a workspace)",
                  p->splits, num_splits, max_blocks, row_bytes * p->splits, cap);
    // automatic choice: the largest split count whose partials fit
    int s = (int)std::min<size_t>((size_t)p->splits, cap / row_bytes);
    for (;; --s) {
      if (s <= 1) {
        p->splits = 1;
        p->pps = max_blocks;
        break;
      }
      st = resolve_splits(pool, S, max_blocks, s, &p->splits, &p->pps);
      if (st) return st;
      if (row_bytes * p->splits <= cap) break;
    }
  }
  // The automatic count s, on a launch of more than one wave: the guided
  // layout (min(2 s, kGuidedSplits) splits whose sizes fall by kGuidedRatio,
  // so the CTAs handed out last, as the grid drains, are short), when its
  // partials fit.  On batches of equal lengths it streams about as fast as s
  // uniform splits (the waves then end together anyway); on ragged ones the
  // drain is what it shortens.
  if (num_splits == 0 && p->splits >= 2) {
    int sms = 0, occ = 0;
    st = decode_residency(pool, &sms, &occ);
    if (st) return st;
    if ((long long)S * pool->desc.n_kv_heads * p->splits > (long long)occ * sms) {
      int b[kGuidedSplits + 1];
      const int n = guided_bounds(max_blocks, std::min(2 * p->splits, kGuidedSplits), b);
      if (n >= 2 && (cap == 0 || row_bytes * n <= cap)) {
        p->guided = true;
        p->splits = n;
        p->pps = b[1];
        for (int i = 0; i <= kGuidedSplits; ++i) p->b[i] = i <= n ? b[i] : max_blocks;
      }
    }
  }
  p->ws_bytes = fixed_ws_bytes(S, n_q_heads, p->splits, D);
  return PA_OK;
}

// pa_decode with a validated plan; `workspace` holds at least plan.ws_bytes.
int decode_with_plan(pa_pool* pool, int layer, void* out, int out_dtype, const void* q,
                     const int32_t* block_tables_dev, int max_blocks_per_seq,
                     const int32_t* ctx_lens_dev, int S, int n_q_heads, float softmax_scale,
                     const Plan& plan, void* workspace, void* stream) {
  const pa_pool_desc& d = pool->desc;
  unsigned int* err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  int dev = 0;
  cudaGetDevice(&dev);
  Dispatch disp = pick(d.kv_dtype, d.head_dim, out_dtype);
  if (configure(*disp.info, dev) <= 0) return fail(PA_ERR_CUDA, "decode kernel configuration failed");
  bool low = false;
  if (plan.bal) {
    if (configure(*disp.info_bal, dev) <= 0) return fail(PA_ERR_CUDA, "decode kernel configuration failed");
  } else if (disp.info_low != disp.info) {
    // A launch that fits one wave of the second build's occupancy takes that
    // build (block-scaled pools: four CTAs per SM without spills, against five).
    const int occ_low = configure(*disp.info_low, dev);
    if (occ_low <= 0) return fail(PA_ERR_CUDA, "decode kernel configuration failed");
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return fail(PA_ERR_CUDA, "SM count query failed");
    low = (long long)S * d.n_kv_heads * plan.splits <= (long long)occ_low * sms;
  }

  const CUtensorMap *tk = nullptr, *tv = nullptr;
  int st = layer_maps(pool, layer, &tk, &tv);
  if (st) return st;

  DecodeArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.out = out;
  a.G = n_q_heads / d.n_kv_heads;
  a.ws_o = static_cast<float*>(workspace);
  if (plan.bal) {
    a.ws_ml = a.ws_o + (size_t)2 * plan.ctas * a.G * d.head_dim;
    a.jobs = reinterpret_cast<int4*>(a.ws_ml + (size_t)2 * plan.ctas * a.G * 2);
  } else {
    a.ws_ml = a.ws_o ? a.ws_o + (size_t)S * n_q_heads * plan.splits * d.head_dim : nullptr;
    a.jobs = nullptr;
  }

  a.tables = block_tables_dev;
  a.ctx = ctx_lens_dev;
  a.max_blocks = max_blocks_per_seq;
  a.S = S;
  a.Hq = n_q_heads;
  a.Hkv = d.n_kv_heads;
  a.num_blocks = d.num_blocks;
  a.splits = plan.splits;
  a.pages_per_split = plan.pps;
  a.sl.splits = plan.splits;
  a.sl.pps = plan.pps;
  a.sl.guided = plan.guided ? 1 : 0;
  for (int i = 0; i <= kGuidedSplits; ++i) a.sl.b[i] = plan.b[i];
  a.ctas = plan.ctas;
  const float log2e = 1.4426950408889634f;
  a.qk_scale_log2 = softmax_scale * log2e * (d.kv_dtype == PA_FP8_E4M3 ? d.k_scale : 1.f);
  a.v_scale = d.kv_dtype == PA_FP8_E4M3 ? d.v_scale : 1.f;
  a.ksc = pool->block_scaled ? layer_scales(pool, pool->k, layer) : nullptr;
  a.vsc = pool->block_scaled ? layer_scales(pool, pool->v, layer) : nullptr;
  a.err = err;
  cudaError_t e = disp.launch(a, tk, tv, S, static_cast<cudaStream_t>(stream), low, plan.bal);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

// Argument checks shared by pa_decode and pa_decode_no_alloc, in the same order.
int check_decode_args(const pa_pool* pool, int layer, int out_dtype, int S, int n_q_heads,
                      int max_blocks_per_seq, float softmax_scale) {
  int st = check_pool_layer(pool, layer);
  if (st) return st;
  st = check_shape(pool, S, n_q_heads, max_blocks_per_seq);
  if (st) return st;
  if (out_dtype != PA_FP32 && out_dtype != in_dtype_of(pool->desc.kv_dtype))
    return fail(PA_ERR_INVALID, "out_dtype must be the query dtype or PA_FP32");
  if (!std::isfinite(softmax_scale)) return fail(PA_ERR_INVALID, "softmax_scale must be finite");
  return PA_OK;
}

int check_decode_ptrs(const void* out, const void* q, const int32_t* tables, const int32_t* ctx) {
  if (!out || !q || !tables || !ctx) return fail(PA_ERR_INVALID, "null argument");
  if (((uintptr_t)out | (uintptr_t)q) & 15u) return fail(PA_ERR_INVALID, "q and out must be 16-byte aligned");
  return PA_OK;
}

int decode_set_wait_limit(unsigned long long ns) { return (int)set_pipe_wait_limit_here(ns); }

}  // namespace pa

using namespace pa;

extern "C" {

int pa_set_pipeline_wait_limit_ns(uint64_t ns) {
  const int e[3] = {decode_set_wait_limit(ns), prefill_set_wait_limit(ns), prefill_tc_set_wait_limit(ns)};
  for (int x : e)
    if (x != (int)cudaSuccess) return fail(PA_ERR_CUDA, "setting the wait limit: %s", cudaGetErrorString((cudaError_t)x));
  return PA_OK;
}

int pa_decode_num_splits(const pa_pool* pool, int S, int n_q_heads, int max_blocks_per_seq,
                         int* num_splits) {
  int st = check_shape(pool, S, n_q_heads, max_blocks_per_seq);
  if (st) return st;
  if (!num_splits) return fail(PA_ERR_INVALID, "null output");
  Plan plan;
  st = make_plan(pool, S, n_q_heads, max_blocks_per_seq, 0, 0, &plan);
  if (st) return st;
  *num_splits = plan.splits;
  return PA_OK;
}

int pa_decode_workspace_bytes(const pa_pool* pool, int S, int n_q_heads, int max_blocks_per_seq,
                              int num_splits, size_t* bytes) {
  int st = check_shape(pool, S, n_q_heads, max_blocks_per_seq);
  if (st) return st;
  if (!bytes) return fail(PA_ERR_INVALID, "null output");
  Plan plan;
  st = make_plan(pool, S, n_q_heads, max_blocks_per_seq, num_splits, 0, &plan);
  if (st) return st;
  *bytes = plan.ws_bytes;
  return PA_OK;
}

int pa_decode(pa_pool* pool, int layer, void* out, int out_dtype, const void* q,
              const int32_t* block_tables_dev, int max_blocks_per_seq, const int32_t* ctx_lens_dev,
              int S, int n_q_heads, float softmax_scale, int num_splits, void* workspace,
              size_t workspace_bytes, void* stream) {
  pa::TraceRange trace_("pa_decode");
  int st = check_decode_args(pool, layer, out_dtype, S, n_q_heads, max_blocks_per_seq, softmax_scale);
  if (st) return st;
  if (num_splits < 0 && num_splits != PA_SPLITS_BALANCED)
    return fail(PA_ERR_INVALID, "num_splits must be >= 0 or PA_SPLITS_BALANCED");
  if (S == 0) return PA_OK;
  st = check_decode_ptrs(out, q, block_tables_dev, ctx_lens_dev);
  if (st) return st;
  Plan plan;
  st = make_plan(pool, S, n_q_heads, max_blocks_per_seq, num_splits, 0, &plan);
  if (st) return st;
  if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes))
    return fail(PA_ERR_INVALID, "workspace of %zu bytes needed (%s), %zu given", plan.ws_bytes,
                plan.bal ? "balanced schedule" : "split partials", workspace_bytes);
  if (plan.ws_bytes > 0 && ((uintptr_t)workspace & 15u))
    return fail(PA_ERR_INVALID, "workspace must be 16-byte aligned");
  return decode_with_plan(pool, layer, out, out_dtype, q, block_tables_dev, max_blocks_per_seq,
                          ctx_lens_dev, S, n_q_heads, softmax_scale, plan, workspace, stream);
}

// ---------------------------------------------------------------------------
// Fixed scratch for pa_decode_no_alloc: the split partials of one call, for
// callers that cannot allocate device memory.  One copy per device that loads
// the library; its device address is looked up once per device and cached for
// the life of the process (a cudaDeviceReset would make the cached address stale).
static __device__ __align__(256) float g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES / sizeof(float)];

static int noalloc_scratch(void** ptr) {
  static std::mutex mu;
  static void* cached[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 128) return fail(PA_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(PA_ERR_CUDA, "cudaGetSymbolAddress(no-alloc scratch): %s", cudaGetErrorString(e));
    cached[dev] = p;
  }
  *ptr = cached[dev];
  return PA_OK;
}

int pa_decode_no_alloc(pa_pool* pool, int layer, void* out, int out_dtype, const void* q,
                       const int32_t* block_tables_dev, int max_blocks_per_seq,
                       const int32_t* ctx_lens_dev, int S, int n_q_heads, float softmax_scale,
                       int num_splits, void* stream) {
  pa::TraceRange trace_("pa_decode_no_alloc");
  int st = check_decode_args(pool, layer, out_dtype, S, n_q_heads, max_blocks_per_seq, softmax_scale);
  if (st) return st;
  if (num_splits < 0 && num_splits != PA_SPLITS_BALANCED)
    return fail(PA_ERR_INVALID, "num_splits must be >= 0 or PA_SPLITS_BALANCED");
  if (S == 0) return PA_OK;
  st = check_decode_ptrs(out, q, block_tables_dev, ctx_lens_dev);
  if (st) return st;
  Plan plan;
  st = make_plan(pool, S, n_q_heads, max_blocks_per_seq, num_splits, PA_NOALLOC_SCRATCH_BYTES, &plan);
  if (st) return st;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);  // also on calls that need none: the lookup happens on the first call
  if (st) return st;
  return decode_with_plan(pool, layer, out, out_dtype, q, block_tables_dev, max_blocks_per_seq,
                          ctx_lens_dev, S, n_q_heads, softmax_scale, plan, scratch, stream);
}

}  // extern "C"
