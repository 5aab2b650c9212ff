// pa_prefill.cu -- chunked prefill attention over the paged KV cache (sm_103a).
//
// Prefill is split into chunks of new tokens that are interleaved with decode
// steps ("Optimización de KV Cache con PagedAttention y Cuantización FP8 para
// Contextos Largos (128K)", sections 5 and 6.3: packets of e.g. 8,192 tokens).
// The chunk's K/V are first written to their slots by pa_reshape_and_cache;
// then each query token of the chunk attends causally to every earlier token
// of its sequence and to itself, reading keys and values page by page through
// the block table ("Capítulo 8 -- Gestión de caché KV de nueva generación",
// section 8.1).
//
// Kernel design (the pages give none):
//  * grid = (16-token query tile, kv head, sequence); tiles are scheduled from
//    the last (longest key range) to the first.  The CTA's rows are the 16
//    tokens x G query heads of the group; each consumer warp owns 16 rows, so a
//    CTA has G consumer warps plus one producer warp.
//  * The producer streams the K and V tiles of pages 0 .. (last query's
//    position) / 16 through the same 8-stage TMA ring as decode; every
//    consumer warp reads every page, so a stage is released after G arrivals.
//  * Per page and warp: S = Q K^T as two m16n8k16 n-tiles (16 rows x 16 keys,
//    fp32 accumulate), the causal mask only on pages that reach the tile's
//    first query, an online softmax per row, and O += P V with P taken
//    straight from the S accumulators (16 dims per n-tile pair).  Q and K share
//    a permutation of the head dim (contiguous 16-byte runs per thread), and the
//    output dims are permuted so each thread reads contiguous runs of V rows.
//  * Block-scaled FP8 pools: each page's K and V scales come with the page (the
//    producer reads them beside the table entries); the K scale joins the
//    softmax exponent's factor, the V scale weights P relative to the largest V
//    scale seen so far, as in decode.
//  * FP8 codes convert exactly to binary16; bf16 q of an FP8 cache is rescaled
//    by a power of two per warp; P is split into two 16-bit parts for bf16
//    caches and the fp32 output mode, as in decode.
//  * The normalised output is staged in shared memory and written row by row.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "pa_device.cuh"

namespace pa {
namespace {

enum { P_F16 = 0, P_BF16 = 1, P_E4M3 = 2, P_E4M3B = 4 };  // P_E4M3B: scale per tile
enum { O_F16 = 0, O_BF16 = 1, O_F32 = 3 };

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kMaxGroup = 8;

template <int KV, int D>
struct PCfg {
  static constexpr bool kFp8 = (KV == P_E4M3) || (KV == P_E4M3B);
  static constexpr bool kBlockScaled = (KV == P_E4M3B);
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kTile = 16 * kRowBytes;
  static constexpr bool kSwizzle = (kRowBytes % 128) == 0;
  static constexpr int kTmaRank = kRowBytes == 256 ? 3 : 2;
  static constexpr int kStages = 8;
  static constexpr int kStageBytes = 2 * kTile;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kStageOut = kMaxGroup * 16 * D * 4;  // output staging, fp32
  static constexpr int kDataBytes = kRingBytes > kStageOut ? kRingBytes : kStageOut;
  static constexpr int kAlign = 1024;
  static constexpr int kScaleBytes = kBlockScaled ? kStages * 8 : 0;  // (K, V) scales per stage
  static constexpr int kSmem = kDataBytes + 2 * kStages * 8 + kScaleBytes + kAlign;
  static constexpr bool kMmaBf16 = (KV == P_BF16);
};

struct PrefillArgs {
  const uint16_t* q;  // [T][Hq][D]
  void* out;          // [T][Hq][D]
  const int32_t* q_start;
  const int32_t* ctx;
  const int32_t* tables;
  int max_blocks;
  int Hq, Hkv, G, num_blocks;
  float qk_scale_log2;
  float v_scale;
  const float* ksc;  // block-scaled pools: this layer's scales [num_blocks][Hkv]
  const float* vsc;
  unsigned int* err;
};

template <int OUT>
__device__ __forceinline__ void store_o(void* out, size_t idx, float v) {
  if constexpr (OUT == O_F32) static_cast<float*>(out)[idx] = v;
  else if constexpr (OUT == O_BF16) static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  else static_cast<__half*>(out)[idx] = __float2half_rn(v);
}

template <int RANK>
__device__ __forceinline__ void load_page_tile(void* dst, const CUtensorMap* map, int row0,
                                               uint64_t* bar, uint64_t policy) {
  if constexpr (RANK == 3) tma_load_3d(dst, map, 0, 0, row0, bar, policy);
  else tma_load_2d(dst, map, 0, row0, bar, policy);
}

template <bool SWZ>
__device__ __forceinline__ uint32_t toff(uint32_t off) {
  if constexpr (SWZ) return swizzle128(off);
  else return off;
}

template <int KV, int D, int OUT, bool PSPLIT>
__global__ void __launch_bounds__((kMaxGroup + 1) * 32) prefill_kernel(
    const PrefillArgs a, const __grid_constant__ CUtensorMap tmk,
    const __grid_constant__ CUtensorMap tmv) {
  using C = PCfg<KV, D>;
  constexpr bool BF = C::kMmaBf16;
  constexpr bool SWZ = C::kSwizzle;
  constexpr bool F8 = C::kFp8;
  constexpr bool BLK = C::kBlockScaled;
  constexpr int NTO = D / 8;  // output n-tiles (8 dims each)
  constexpr int QW = D / 8;   // 32-bit words of q per row per thread
  constexpr int KB = D / 4 * C::kElem;
  constexpr int VB = D / 8 * C::kElem;
  constexpr int RB = C::kRowBytes;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + C::kAlign - 1) & ~uintptr_t(C::kAlign - 1));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kDataBytes);
  uint64_t* empty = full + C::kStages;
  float2* stage_scale = reinterpret_cast<float2*>(smem + C::kDataBytes + 2 * C::kStages * 8);

  const int qt = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, seq = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G;
  const int q0 = a.q_start[seq];
  const int Cn = a.q_start[seq + 1] - q0;
  // a negative start or a decreasing pair: the sequence is skipped
  if (q0 < 0 || Cn < 0) {
    if (threadIdx.x == 0) record_error(a.err, PA_ERR_BOUNDS);
    return;
  }
  // a chunk longer than the grid covers (max_chunk): its rows past the grid
  // are not written; the CTA of the last tile reports it
  if (qt == (int)gridDim.x - 1 && Cn > 16 * (int)gridDim.x && threadIdx.x == 0)
    record_error(a.err, PA_ERR_BOUNDS);
  const int tok_lo = 16 * qt;
  if (tok_lo >= Cn) return;
  const int ctx = a.ctx[seq];
  if (ctx < Cn || ctx > a.max_blocks * 16) {
    if (threadIdx.x == 0) record_error(a.err, PA_ERR_BOUNDS);
    return;
  }
  const int n_tok = min(16, Cn - tok_lo);
  const int pos0 = ctx - Cn + tok_lo;  // position of the tile's first query
  const int pos_last = pos0 + n_tok - 1;
  const int npages = pos_last / 16 + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], G);
    }
    fence_barrier_init();
  }
  if (threadIdx.x == G * 32) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  __syncthreads();

  if (warp == G) {
    // ------------------------------------------------------------ producer
    const int32_t* trow = a.tables + (size_t)seq * a.max_blocks;
    const uint64_t policy = l2_evict_first_policy();
    int issued = 0;
    bool abort = false;
    for (int base = 0; base < npages && !abort; base += 32) {
      int phys = 0;
      float sk = 0.f, sv = 0.f;
      if (base + lane < npages) {
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
      const int cnt = min(32, npages - base);
      for (int j = 0; j < cnt; ++j) {
        const int ph = __shfl_sync(kFullMask, phys, j);
        float skj = 0.f, svj = 0.f;
        if constexpr (BLK) {
          skj = __shfl_sync(kFullMask, sk, j);
          svj = __shfl_sync(kFullMask, sv, j);
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
            if constexpr (BLK) stage_scale[stage] = make_float2(skj, svj);  // published by the arrive
            mbar_arrive_expect_tx(&full[stage], 2 * C::kTile);
            load_page_tile<C::kTmaRank>(dst, &tmk, row0, &full[stage], policy);
            load_page_tile<C::kTmaRank>(dst + C::kTile, &tmv, row0, &full[stage], policy);
            ++issued;
          }
        }
        if (__shfl_sync(kFullMask, stop, 0)) {
          abort = true;
          break;
        }
      }
    }
    if (lane == 0) {
      for (int s = 0; s < C::kStages && s < issued; ++s) {
        const int uses = (issued - 1 - s) / C::kStages + 1;
        if (!mbar_wait(&full[s], (uses - 1) & 1)) record_error(a.err, PA_ERR_TIMEOUT);
      }
    }
    __syncthreads();  // matches the consumers' barrier before the output staging
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  // rows of this warp: r = 16 * warp + g (+ 8); row r is token r / G, head r % G
  const int r0 = 16 * warp + g, r1 = r0 + 8;
  const int tl0 = r0 / G, hh0 = r0 - tl0 * G;
  const int tl1 = r1 / G, hh1 = r1 - tl1 * G;
  const bool v0 = tl0 < n_tok, v1 = tl1 < n_tok;
  const int qp0 = pos0 + min(tl0, n_tok - 1);  // causal limit of each row
  const int qp1 = pos0 + min(tl1, n_tok - 1);

  uint32_t qa0[QW], qa1[QW];  // rows r0, r1: dims [t*D/4, (t+1)*D/4) as 16-bit pairs
  float qk_scale = a.qk_scale_log2;
  {
    uint32_t raw0[QW], raw1[QW];
    const uint16_t* base = a.q + ((size_t)(q0 + tok_lo) * a.Hq + (size_t)h * G) * D + t * (D / 4);
    const uint4* s0 = reinterpret_cast<const uint4*>(base + ((size_t)tl0 * a.Hq + hh0) * D);
    const uint4* s1 = reinterpret_cast<const uint4*>(base + ((size_t)tl1 * a.Hq + hh1) * D);
#pragma unroll
    for (int c = 0; c < QW / 4; ++c) {
      const uint4 u0 = v0 ? s0[c] : make_uint4(0, 0, 0, 0);
      const uint4 u1 = v1 ? s1[c] : make_uint4(0, 0, 0, 0);
      raw0[4 * c] = u0.x; raw0[4 * c + 1] = u0.y; raw0[4 * c + 2] = u0.z; raw0[4 * c + 3] = u0.w;
      raw1[4 * c] = u1.x; raw1[4 * c + 1] = u1.y; raw1[4 * c + 2] = u1.z; raw1[4 * c + 3] = u1.w;
    }
    if constexpr (F8) {
      float amax = 0.f;
#pragma unroll
      for (int w = 0; w < QW; ++w) {
        amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(raw0[w] & 0xFFFFu)),
                                 fabsf(bf16_bits_to_float(raw0[w] >> 16))));
        amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(raw1[w] & 0xFFFFu)),
                                 fabsf(bf16_bits_to_float(raw1[w] >> 16))));
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1)
        amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, off));
      int ex = 0;
      if (amax > 0.f) frexpf(amax, &ex);
      const float qs = amax > 0.f ? ldexpf(1.f, 15 - ex) : 1.f;
      qk_scale = amax > 0.f ? qk_scale * ldexpf(1.f, ex - 15) : qk_scale;
#pragma unroll
      for (int w = 0; w < QW; ++w) {
        qa0[w] = pack2<false>(bf16_bits_to_float(raw0[w] & 0xFFFFu) * qs,
                              bf16_bits_to_float(raw0[w] >> 16) * qs);
        qa1[w] = pack2<false>(bf16_bits_to_float(raw1[w] & 0xFFFFu) * qs,
                              bf16_bits_to_float(raw1[w] >> 16) * qs);
      }
    } else {
#pragma unroll
      for (int w = 0; w < QW; ++w) {
        qa0[w] = raw0[w];
        qa1[w] = raw1[w];
      }
    }
  }

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[NTO][4];
#pragma unroll
  for (int i = 0; i < NTO; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  // block-scaled pools: V weights relative to the largest V scale seen (as in decode)
  float vref = 0.f, vref_inv = 0.f;

  for (int k = 0; k < npages; ++k) {
    const int stage = k % C::kStages;
    if (!__all_sync(kFullMask, mbar_wait(&full[stage], (k / C::kStages) & 1, pipe_wait_limit()))) {
      if (lane == 0) record_error(a.err, PA_ERR_TIMEOUT);
      break;
    }
    const uint8_t* Ks = ring + stage * C::kStageBytes;
    const uint8_t* Vs = Ks + C::kTile;
    const int key0 = 16 * k;
    float2 psc = make_float2(1.f, 1.f);
    if constexpr (BLK) psc = stage_scale[stage];

    // ---- S[row][key] = Q K^T, keys g + 8 nt of this page per n-tile nt
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      const uint32_t kro = (g + 8 * nt) * RB + t * KB;
#pragma unroll
      for (int c = 0; c < KB / 16; ++c) {
        const uint4 r = lds128(Ks + toff<SWZ>(kro + 16 * c));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
        if constexpr (F8) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = 4 * c + jj;  // dims t*D/4 + 4j .. 4j+3
            const uint32_t af[4] = {qa0[2 * j], qa1[2 * j], qa0[2 * j + 1], qa1[2 * j + 1]};
            uint32_t b0, b1;
            e4m3x4_to_f16x2x2(w[jj], b0, b1);
            mma16816<false>(s[nt], af, b0, b1);
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int j = 2 * c + jj;
            const uint32_t af[4] = {qa0[2 * j], qa1[2 * j], qa0[2 * j + 1], qa1[2 * j + 1]};
            mma16816<BF>(s[nt], af, w[2 * jj], w[2 * jj + 1]);
          }
        }
      }
    }

    // ---- causal mask (pages that reach the tile's first query) and online softmax
    float x[2][4];
    const float qks = BLK ? qk_scale * psc.x : qk_scale;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[nt][e] = s[nt][e] * qks;
    if (key0 + 15 > pos0) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int kp = key0 + 8 * nt + 2 * t;
        if (kp > qp0) x[nt][0] = -INFINITY;
        if (kp + 1 > qp0) x[nt][1] = -INFINITY;
        if (kp > qp1) x[nt][2] = -INFINITY;
        if (kp + 1 > qp1) x[nt][3] = -INFINITY;
      }
    }
    float pm0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
    float pm1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      pm0 = fmaxf(pm0, __shfl_xor_sync(kFullMask, pm0, off));
      pm1 = fmaxf(pm1, __shfl_xor_sync(kFullMask, pm1, off));
    }
    // key 0 (page 0) is visible to every row, so the maxima are finite from there on
    const float mn0 = fmaxf(m0, pm0), mn1 = fmaxf(m1, pm1);
    const bool vgrow = BLK && psc.y > vref;  // warp-uniform
    if (__any_sync(kFullMask, (mn0 != m0) | (mn1 != m1)) || vgrow) {
      const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
      l0 *= al0;
      l1 *= al1;
      float ov0 = al0, ov1 = al1;
      if constexpr (BLK) {
        if (vgrow) {
          const float r = vref / psc.y;
          ov0 *= r;
          ov1 *= r;
          vref = psc.y;
          vref_inv = 1.f / psc.y;
        }
      }
#pragma unroll
      for (int i = 0; i < NTO; ++i) {
        o[i][0] *= ov0;
        o[i][1] *= ov0;
        o[i][2] *= ov1;
        o[i][3] *= ov1;
      }
      m0 = mn0;
      m1 = mn1;
    }
    float p[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      p[nt][0] = fast_exp2(x[nt][0] - m0);
      p[nt][1] = fast_exp2(x[nt][1] - m0);
      p[nt][2] = fast_exp2(x[nt][2] - m1);
      p[nt][3] = fast_exp2(x[nt][3] - m1);
      l0 += p[nt][0] + p[nt][1];
      l1 += p[nt][2] + p[nt][3];
    }
    if constexpr (BLK) {  // weights of this page's V codes: P * sv / vref
      const float f = psc.y * vref_inv;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) p[nt][e] *= f;
    }
    // P as the A operand: rows g / g+8, keys 2t,2t+1 (a0,a1) and 2t+8,2t+9 (a2,a3)
    uint32_t pa[4] = {pack2<BF>(p[0][0], p[0][1]), pack2<BF>(p[0][2], p[0][3]),
                      pack2<BF>(p[1][0], p[1][1]), pack2<BF>(p[1][2], p[1][3])};
    uint32_t pr[4] = {0, 0, 0, 0};
    if constexpr (PSPLIT) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 u = unpack2<BF>(pa[i]);
        const int nt = i >> 1, e = (i & 1) * 2;
        pr[i] = pack2<BF>(p[nt][e] - u.x, p[nt][e + 1] - u.y);
      }
    }

    // ---- O[row][dim] += P V; B column n = g of n-tile nt is dim g * D/8 + nt
    {
      const int rows[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
      constexpr int VW = VB / 4;
      uint32_t vw[4][VW];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t vo = rows[r] * RB + g * VB;
        if constexpr (VB == 8) {
          const uint2 u = lds64(Vs + toff<SWZ>(vo));
          vw[r][0] = u.x;
          vw[r][1] = u.y;
        } else {
#pragma unroll
          for (int c = 0; c < VB / 16; ++c) {
            const uint4 u = lds128(Vs + toff<SWZ>(vo + 16 * c));
            vw[r][4 * c] = u.x;
            vw[r][4 * c + 1] = u.y;
            vw[r][4 * c + 2] = u.z;
            vw[r][4 * c + 3] = u.w;
          }
        }
      }
      if (key0 + 15 > pos_last) {  // slots past the last query may hold anything
#pragma unroll
        for (int r = 0; r < 4; ++r)
          if (key0 + rows[r] > pos_last) {
#pragma unroll
            for (int w = 0; w < VW; ++w) vw[r][w] = 0u;
          }
      }
#pragma unroll
      for (int nt = 0; nt < NTO; ++nt) {
        uint32_t b0, b1;
        if constexpr (F8) {
          const int w = nt >> 2, e = nt & 3;
          const uint32_t sel = (e < 2) ? 0x5140u : 0x7362u;
          const uint32_t x01 = __byte_perm(vw[0][w], vw[1][w], sel);
          const uint32_t x23 = __byte_perm(vw[2][w], vw[3][w], sel);
          uint32_t l0, h0, l1, h1;
          e4m3x4_to_f16x2x2(x01, l0, h0);
          e4m3x4_to_f16x2x2(x23, l1, h1);
          b0 = (e & 1) ? h0 : l0;
          b1 = (e & 1) ? h1 : l1;
        } else {
          const int w = nt >> 1;
          const uint32_t sel = (nt & 1) ? 0x7632u : 0x5410u;
          b0 = __byte_perm(vw[0][w], vw[1][w], sel);
          b1 = __byte_perm(vw[2][w], vw[3][w], sel);
        }
        mma16816<BF>(o[nt], pa, b0, b1);
        if constexpr (PSPLIT) mma16816<BF>(o[nt], pr, b0, b1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }

#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l0 += __shfl_xor_sync(kFullMask, l0, off);
    l1 += __shfl_xor_sync(kFullMask, l1, off);
  }
  __syncthreads();  // every warp is done with the ring: stage the output there

  // stage rows g / g+8: accumulator column c of n-tile nt is dim c * D/8 + nt
  float* st = reinterpret_cast<float*>(smem) + warp * 16 * D;
  const float vs = BLK ? vref : a.v_scale;
  const float i0 = l0 > 0.f ? vs / l0 : 0.f;
  const float i1 = l1 > 0.f ? vs / l1 : 0.f;
  const int c0 = (2 * t) * (D / 8), c1 = (2 * t + 1) * (D / 8);
#pragma unroll
  for (int nt = 0; nt < NTO; ++nt) {
    st[g * D + c0 + nt] = o[nt][0] * i0;
    st[g * D + c1 + nt] = o[nt][1] * i0;
    st[(g + 8) * D + c0 + nt] = o[nt][2] * i1;
    st[(g + 8) * D + c1 + nt] = o[nt][3] * i1;
  }
  __syncwarp();
  for (int rr = 0; rr < 16; ++rr) {
    const int r = 16 * warp + rr, tl = r / G, hh = r - tl * G;
    if (tl >= n_tok) continue;
    const size_t orow = ((size_t)(q0 + tok_lo + tl) * a.Hq + (size_t)h * G + hh) * D;
    for (int d = lane; d < D; d += 32) store_o<OUT>(a.out, orow + d, st[rr * D + d]);
  }
}

struct PInfo {
  const void* fn;
  int smem;
  bool configured[128];
};

template <int KV, int D, int OUT>
struct PLauncher {
  static constexpr bool kPsplit = (KV == P_BF16) || (OUT == O_F32);
  static PInfo& info() {
    static PInfo pi = {reinterpret_cast<const void*>(&prefill_kernel<KV, D, OUT, kPsplit>),
                       PCfg<KV, D>::kSmem, {}};
    return pi;
  }
  static cudaError_t launch(const PrefillArgs& a, const CUtensorMap* tk, const CUtensorMap* tv,
                            int tiles, int S, cudaStream_t st) {
    dim3 grid(tiles, a.Hkv, S);
    prefill_kernel<KV, D, OUT, kPsplit>
        <<<grid, (a.G + 1) * 32, PCfg<KV, D>::kSmem, st>>>(a, *tk, *tv);
    return cudaGetLastError();
  }
};

struct PDispatch {
  PInfo* info;
  cudaError_t (*launch)(const PrefillArgs&, const CUtensorMap*, const CUtensorMap*, int, int,
                        cudaStream_t);
};

template <int KV, int D, int OUT>
PDispatch pmake() {
  return {&PLauncher<KV, D, OUT>::info(), &PLauncher<KV, D, OUT>::launch};
}

template <int KV, int D>
PDispatch ppick_out(int out_dtype) {
  if (out_dtype == PA_FP32) return pmake<KV, D, O_F32>();
  if constexpr (KV == P_F16) return pmake<KV, D, O_F16>();
  else return pmake<KV, D, O_BF16>();
}

PDispatch ppick(int kv_dtype, int head_dim, int out_dtype) {
  const bool d64 = head_dim == 64;
  switch (kv_dtype) {
    case PA_FP16:
      return d64 ? ppick_out<P_F16, 64>(out_dtype) : ppick_out<P_F16, 128>(out_dtype);
    case PA_BF16:
      return d64 ? ppick_out<P_BF16, 64>(out_dtype) : ppick_out<P_BF16, 128>(out_dtype);
    case PA_FP8_E4M3_BLOCK:
      return d64 ? ppick_out<P_E4M3B, 64>(out_dtype) : ppick_out<P_E4M3B, 128>(out_dtype);
    default:
      return d64 ? ppick_out<P_E4M3, 64>(out_dtype) : ppick_out<P_E4M3, 128>(out_dtype);
  }
}

int pconfigure(PInfo& pi) {
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!pi.configured[dev]) {
    if (cudaFuncSetAttribute(pi.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, pi.smem) !=
        cudaSuccess)
      return 0;
    pi.configured[dev] = true;
  }
  return 1;
}

}  // namespace
int prefill_set_wait_limit(unsigned long long ns) { return (int)set_pipe_wait_limit_here(ns); }

}  // namespace pa

using namespace pa;

extern "C" {

int pa_prefill(pa_pool* pool, int layer, void* out, int out_dtype, const void* q,
               const int32_t* q_start_dev, const int32_t* block_tables_dev, int max_blocks_per_seq,
               const int32_t* ctx_lens_dev, int S, int n_q_heads, int max_chunk,
               float softmax_scale, void* stream) {
  pa::TraceRange trace_("pa_prefill");
  int st = check_pool_layer(pool, layer);
  if (st) return st;
  const pa_pool_desc& d = pool->desc;
  if (S < 0 || max_blocks_per_seq < 1 || n_q_heads < 1 || max_chunk < 0)
    return fail(PA_ERR_INVALID, "need S >= 0, max_blocks_per_seq >= 1, n_q_heads >= 1, max_chunk >= 0");
  if (n_q_heads % d.n_kv_heads != 0)
    return fail(PA_ERR_INVALID, "n_q_heads %d is not a multiple of n_kv_heads %d", n_q_heads,
                d.n_kv_heads);
  const int G = n_q_heads / d.n_kv_heads;
  if (G > kMaxGroup)
    return fail(PA_ERR_UNSUPPORTED, "query heads per kv head must be <= 8 (got %d)", G);
  const int in_dtype = d.kv_dtype == PA_FP16 ? PA_FP16 : PA_BF16;
  if (out_dtype != PA_FP32 && out_dtype != in_dtype)
    return fail(PA_ERR_INVALID, "out_dtype must be the query dtype or PA_FP32");
  if (!std::isfinite(softmax_scale)) return fail(PA_ERR_INVALID, "softmax_scale must be finite");
  if (S == 0 || max_chunk == 0) return PA_OK;
  if (S > 65535 || d.n_kv_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "grid too large");
  if (!out || !q || !q_start_dev || !block_tables_dev || !ctx_lens_dev)
    return fail(PA_ERR_INVALID, "null argument");
  if (((uintptr_t)out | (uintptr_t)q) & 15u) return fail(PA_ERR_INVALID, "q and out must be 16-byte aligned");
  unsigned int* err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  if (prefill_tc_supported(pool, n_q_heads, out_dtype))
    return prefill_tc(pool, layer, out, out_dtype, q, q_start_dev, block_tables_dev, max_blocks_per_seq,
                      ctx_lens_dev, S, n_q_heads, max_chunk, softmax_scale, err,
                      static_cast<cudaStream_t>(stream));
  PDispatch disp = ppick(d.kv_dtype, d.head_dim, out_dtype);
  if (!pconfigure(*disp.info)) return fail(PA_ERR_CUDA, "prefill kernel configuration failed");
  const CUtensorMap_st *tk = nullptr, *tv = nullptr;
  st = layer_maps(pool, layer, &tk, &tv);
  if (st) return st;
  PrefillArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.out = out;
  a.q_start = q_start_dev;
  a.ctx = ctx_lens_dev;
  a.tables = block_tables_dev;
  a.max_blocks = max_blocks_per_seq;
  a.Hq = n_q_heads;
  a.Hkv = d.n_kv_heads;
  a.G = G;
  a.num_blocks = d.num_blocks;
  a.qk_scale_log2 = softmax_scale * 1.4426950408889634f * (d.kv_dtype == PA_FP8_E4M3 ? d.k_scale : 1.f);
  a.v_scale = d.kv_dtype == PA_FP8_E4M3 ? d.v_scale : 1.f;
  a.ksc = pool->block_scaled ? layer_scales(pool, pool->k, layer) : nullptr;
  a.vsc = pool->block_scaled ? layer_scales(pool, pool->v, layer) : nullptr;
  a.err = err;
  const int tiles = (max_chunk + 15) / 16;
  cudaError_t e = disp.launch(a, tk, tv, tiles, S, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

}  // extern "C"
