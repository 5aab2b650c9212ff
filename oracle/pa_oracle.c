/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for paged KV-cache decode.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline / reference leg may load this code.  It
 * shares no header, helper, table or constant with the CUDA library: every
 * format, layout and formula below is written out again from its definition.
 *
 * What it computes, and where that is stated:
 *
 *  - Bytes per token of a KV cache, 2 * n_layers * n_kv_heads * d_head * bytes
 *    ("Optimización de KV Cache con PagedAttention y Cuantización FP8 para
 *    Contextos Largos (128K)", section 2).
 *  - A flat pool of fixed-size blocks (16 tokens) addressed through a per-
 *    sequence block table: logical block j of a sequence lives in physical
 *    block table[j] ("Capítulo 8 -- Gestión de caché KV de nueva generación",
 *    section 8.1; "PagedAttention y Gestión de KV-Cache", section 2 figure).
 *    Pool layout, per layer: K and V separate, each [num_blocks][n_kv_heads]
 *    [block_size][head_dim] elements.
 *  - Writing a new token's K/V into its slot (slot = block * block_size +
 *    offset), converting 16-bit values to 8-bit FP8 on the fly when the cache is
 *    FP8 ("Optimización de KV Cache ...", section 4).  FP8 is OCP E4M3FN:
 *    code = e4m3_rne_satfinite( fl32(x / scale) ), with a static per-tensor
 *    scale (same page, section 8, static calibration).
 *  - Decode attention: gather a sequence's pages in logical order into
 *    contiguous K, V, then textbook softmax attention per query head, with
 *    query head g reading kv head floor(g / G), G = n_q_heads / n_kv_heads.
 *    Everything in fp64.  A sequence of context length 0 yields a zero output.
 *  - Chunked prefill: a chunk of C new tokens of a sequence, already written
 *    to the cache, each attend causally to every earlier token and to
 *    themselves (prefill split into packets interleaved with decode steps,
 *    "Optimización de KV Cache ...", sections 5 and 6.3).  Query j of a chunk
 *    that ends the sequence's ctx tokens sits at position ctx - C + j and sees
 *    tokens [0, ctx - C + j].
 *  - Dynamic per-block FP8 scaling (same page, section 8, dynamic scaling:
 *    the MaxAbs of each block is taken at inference time and the scale is
 *    applied on the fly).  Each (block, kv head) tile of K, and of V, has its
 *    own fp32 scale s = fl32(MaxAbs / 448), 448 being the largest E4M3 value;
 *    s = 0 marks a tile whose values are all zero (its codes are then 0).
 *    The page does not say how a block that fills token by token keeps its
 *    MaxAbs; the reading taken here: the tokens one call writes into a block
 *    form one run of consecutive slots; a run that starts at offset 0 starts
 *    the tile afresh; a later run that raises the tile's MaxAbs re-encodes the
 *    tile's earlier rows with the new scale, from their dequantised fp32
 *    values (the 16-bit originals are no longer held).  Pool regions of this
 *    type are the code tiles followed by the scale table
 *    [num_blocks][n_kv_heads] of fp32.
 *  - Swap of whole blocks to host memory: the K and V tiles of every kv head
 *    of a block, block after block ("KV Cache y PagedAttention", fine-grained
 *    eviction of pages to the CPU).
 *  - Copy of whole blocks (K and V tiles of every kv head), the copy-on-write
 *    step of shared prefixes ("PagedAttention y Gestión de KV-Cache", section
 *    3.01; "KV Cache y PagedAttention", "Cómo PagedAttention soluciona esto").
 *
 * Dtype codes used by this file (its own, passed in by its Python wrapper):
 *   0 = IEEE binary16, 1 = bfloat16, 2 = FP8 E4M3FN with per-tensor scales,
 *   3 = FP8 E4M3FN with a dynamic scale per (block, kv head) tile.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F16 0
#define OR_BF16 1
#define OR_E4M3 2
#define OR_E4M3_BLK 3

/* ---------------------------------------------------------------------------
 * Number formats, decoded from their bit-level definitions.
 * ------------------------------------------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double or_f16_value(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 10) & 0x1F;
  int f = bits & 0x3FF;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
  } else if (e == 31) {
    v = (f == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double or_bf16_value(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3FN: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * No infinities; S.1111.111 is NaN; exponent field 0 holds subnormals
 * m * 2^-9; largest finite value 1.75 * 2^8 = 448. */
double or_e4m3_value(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) {
    v = ldexp((double)m, -9);
  } else {
    v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  }
  return sign ? -v : v;
}

/* Round a non-negative real q to an integer, ties to the even integer. */
static double round_half_even(double q) {
  double fl = floor(q);
  double r = q - fl; /* exact: q has at most 53 significant bits */
  if (r > 0.5) return fl + 1.0;
  if (r < 0.5) return fl;
  return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* E4M3 encoding of an fp32 value y: round to the nearest point of the E4M3
 * grid, ties to the even mantissa (subnormals included), then saturate any
 * magnitude above 448 to 448 ("satfinite").  The sign is kept, so -0 -> 0x80.
 * NaN maps to 0x7F (this case is outside every workload here). */
uint8_t or_e4m3_encode(float y) {
  if (isnan(y)) return 0x7F;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormal binade: grid step 2^-9; n == 8 is the smallest normal 2^-6,
     * whose code (exponent 1, mantissa 0) is also 8. */
    double n = round_half_even(a * 512.0);
    return sign | (uint8_t)n;
  }
  int k;
  frexp(a, &k); /* a = f * 2^k, f in [0.5, 1): a lies in binade 2^(k-1) */
  int ebin = k - 1;                 /* unbiased exponent, -6 .. 8 */
  double step = ldexp(1.0, ebin - 3); /* 3 mantissa bits */
  double n = round_half_even(a / step); /* in [8, 16]; 16 carries up a binade */
  int code = ((ebin + 7) << 3) + ((int)n - 8);
  if (code > 0x7E) code = 0x7E; /* cannot happen for a < 448; kept for clarity */
  return sign | (uint8_t)code;
}

/* Quantise one stored 16-bit value x with the per-tensor scale s:
 * y = fl32(x / s) (the fp64 quotient rounded once to fp32 equals the IEEE fp32
 * quotient, since 53 >= 2*24 + 2), then E4M3 with saturation. */
uint8_t or_quantize_e4m3(double x, float s) {
  float y = (float)(x / (double)s);
  return or_e4m3_encode(y);
}

double or_value16(int dtype, uint16_t bits) {
  return dtype == OR_BF16 ? or_bf16_value(bits) : or_f16_value(bits);
}

/* Closed form of the KV-cache size per token (one K and one V vector per kv
 * head per layer). */
long long or_kv_bytes_per_token(int n_layers, int n_kv_heads, int d_head, int precision_bytes) {
  return 2LL * n_layers * n_kv_heads * d_head * precision_bytes;
}

/* Bytes of one element of the pool for a cache dtype. */
static int elem_bytes(int kv_dtype) { return (kv_dtype == OR_E4M3 || kv_dtype == OR_E4M3_BLK) ? 1 : 2; }

/* Bytes of the code tiles of one K or V region: [num_blocks][n_kv_heads]
 * [block_size][head_dim] elements.  A block-scaled region continues with its
 * scale table right after them. */
static long long tiles_bytes(int kv_dtype, int num_blocks, int n_kv_heads, int block_size,
                             int head_dim) {
  return (long long)num_blocks * n_kv_heads * block_size * head_dim * elem_bytes(kv_dtype);
}

/* Scale of tile (block, h) of a block-scaled region, and its update. */
static float tile_scale_get(const uint8_t* pool, long long tiles, int n_kv_heads, int block, int h) {
  float s;
  memcpy(&s, pool + tiles + 4 * ((long long)block * n_kv_heads + h), 4);
  return s;
}
static void tile_scale_set(uint8_t* pool, long long tiles, int n_kv_heads, int block, int h, float s) {
  memcpy(pool + tiles + 4 * ((long long)block * n_kv_heads + h), &s, 4);
}

/* Element index of (block, kv head, offset within block, dim) in one layer's
 * K or V pool of layout [num_blocks][n_kv_heads][block_size][head_dim]. */
static long long pool_index(int block, int h, int off, int i, int n_kv_heads, int block_size,
                            int head_dim) {
  return (((long long)block * n_kv_heads + h) * block_size + off) * head_dim + i;
}

/* Value of pool element idx (already dequantised for FP8). */
static double pool_value(int kv_dtype, const uint8_t* pool, long long idx, float scale) {
  if (kv_dtype == OR_E4M3 || kv_dtype == OR_E4M3_BLK) return or_e4m3_value(pool[idx]) * (double)scale;
  uint16_t bits;
  memcpy(&bits, pool + 2 * idx, 2);
  return or_value16(kv_dtype, bits);
}

/* ---------------------------------------------------------------------------
 * Dynamic per-block scaling of one run of n tokens (rows off0 .. off0+n-1 of
 * tile (block, h)) of one tensor, K or V.  x: the run's values, row r at
 * x[r * ld .. r * ld + head_dim).  The tile's scale follows its MaxAbs:
 *   m     = max |x| over the run (exact: 16-bit values)
 *   s_run = fl32(m / 448)
 *   off0 == 0 : s = s_run (the tile starts afresh)
 *   off0 >  0 : s = max(s_old, s_run); if s > s_old, each earlier code c of
 *               rows 0 .. off0-1 becomes E4M3(fl32(fl32(value(c) * s_old) / s))
 * then each new value is stored as E4M3(fl32(x / s)) (code 0 when s = 0). */
static void write_run_block_scaled(const double* x, long long ld, int n, int off0, int block, int h,
                                   int n_kv_heads, int block_size, int head_dim, long long tiles,
                                   uint8_t* pool) {
  double m = 0.0;
  for (int r = 0; r < n; ++r)
    for (int i = 0; i < head_dim; ++i)
      if (fabs(x[r * ld + i]) > m) m = fabs(x[r * ld + i]);
  float s = (float)(m / 448.0);
  if (off0 > 0) {
    float s_old = tile_scale_get(pool, tiles, n_kv_heads, block, h);
    if (s > s_old) {
      for (int r = 0; r < off0; ++r)
        for (int i = 0; i < head_dim; ++i) {
          long long idx = pool_index(block, h, r, i, n_kv_heads, block_size, head_dim);
          float y_old = (float)(or_e4m3_value(pool[idx]) * (double)s_old);
          pool[idx] = or_quantize_e4m3((double)y_old, s);
        }
    } else {
      s = s_old;
    }
  }
  for (int r = 0; r < n; ++r)
    for (int i = 0; i < head_dim; ++i) {
      long long idx = pool_index(block, h, off0 + r, i, n_kv_heads, block_size, head_dim);
      pool[idx] = s > 0.f ? or_quantize_e4m3(x[r * ld + i], s) : 0x00;
    }
  tile_scale_set(pool, tiles, n_kv_heads, block, h, s);
}

/* reshape_and_cache of a block-scaled FP8 pool: tokens are taken in runs --
 * a token, then the tokens right after it in slot_mapping whose slots follow
 * it within the same block -- and each run updates its tiles as above.  (The
 * tokens one call writes into a block are expected to form a single run.) */
static int reshape_block_scaled(int num_blocks, int block_size, int n_kv_heads, int head_dim,
                                const uint16_t* k_in, const uint16_t* v_in,
                                const int64_t* slot_mapping, int T, uint8_t* k_pool,
                                uint8_t* v_pool) {
  int status = 0;
  long long tiles = tiles_bytes(OR_E4M3_BLK, num_blocks, n_kv_heads, block_size, head_dim);
  long long row = (long long)n_kv_heads * head_dim;
  double* xk = (double*)malloc(sizeof(double) * (size_t)(block_size * head_dim));
  double* xv = (double*)malloc(sizeof(double) * (size_t)(block_size * head_dim));
  int t = 0;
  while (t < T) {
    int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= (int64_t)num_blocks * block_size) {
      if (slot >= 0) status = -1;
      ++t;
      continue;
    }
    int block = (int)(slot / block_size), off0 = (int)(slot % block_size);
    int n = 1;
    while (t + n < T && off0 + n < block_size && slot_mapping[t + n] == slot + n) ++n;
    for (int h = 0; h < n_kv_heads; ++h) {
      for (int r = 0; r < n; ++r)
        for (int i = 0; i < head_dim; ++i) {
          long long src = (t + r) * row + (long long)h * head_dim + i;
          xk[r * head_dim + i] = or_bf16_value(k_in[src]);
          xv[r * head_dim + i] = or_bf16_value(v_in[src]);
        }
      write_run_block_scaled(xk, head_dim, n, off0, block, h, n_kv_heads, block_size, head_dim,
                             tiles, k_pool);
      write_run_block_scaled(xv, head_dim, n, off0, block, h, n_kv_heads, block_size, head_dim,
                             tiles, v_pool);
    }
    t += n;
  }
  free(xk);
  free(xv);
  return status;
}

/* ---------------------------------------------------------------------------
 * Writing new tokens into their slots.
 *   k_in, v_in : [T][n_kv_heads][head_dim] 16-bit bit patterns (input dtype:
 *                binary16 for a binary16 cache, bfloat16 otherwise)
 *   slot_mapping[t] = block * block_size + offset, or negative to skip token t
 * Returns 0, or -1 if some slot lies beyond the pool (nothing is written for it).
 * ------------------------------------------------------------------------- */
int or_reshape_and_cache(int kv_dtype, int num_blocks, int block_size, int n_kv_heads,
                         int head_dim, const uint16_t* k_in, const uint16_t* v_in,
                         const int64_t* slot_mapping, int T, float k_scale, float v_scale,
                         uint8_t* k_pool, uint8_t* v_pool) {
  if (kv_dtype == OR_E4M3_BLK)
    return reshape_block_scaled(num_blocks, block_size, n_kv_heads, head_dim, k_in, v_in,
                                slot_mapping, T, k_pool, v_pool);
  int status = 0;
  int in_dtype = (kv_dtype == OR_F16) ? OR_F16 : OR_BF16;
  for (int t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= (int64_t)num_blocks * block_size) {
      status = -1;
      continue;
    }
    int block = (int)(slot / block_size);
    int off = (int)(slot % block_size);
    for (int h = 0; h < n_kv_heads; ++h) {
      for (int i = 0; i < head_dim; ++i) {
        long long src = ((long long)t * n_kv_heads + h) * head_dim + i;
        long long dst = pool_index(block, h, off, i, n_kv_heads, block_size, head_dim);
        if (kv_dtype == OR_E4M3) {
          k_pool[dst] = or_quantize_e4m3(or_value16(in_dtype, k_in[src]), k_scale);
          v_pool[dst] = or_quantize_e4m3(or_value16(in_dtype, v_in[src]), v_scale);
        } else {
          memcpy(k_pool + 2 * dst, &k_in[src], 2);
          memcpy(v_pool + 2 * dst, &v_in[src], 2);
        }
      }
    }
  }
  return status;
}

/* Copy whole blocks: for each pair (src, dst), the K and V tiles of every kv
 * head of one layer.  pairs: [n][2].  Returns -1 if an id is out of range. */
int or_copy_blocks(int kv_dtype, int num_blocks, int block_size, int n_kv_heads, int head_dim,
                   const int32_t* pairs, int n, uint8_t* k_pool, uint8_t* v_pool) {
  long long blk = (long long)n_kv_heads * block_size * head_dim * elem_bytes(kv_dtype);
  int status = 0;
  for (int p = 0; p < n; ++p) {
    int src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      status = -1;
      continue;
    }
    memmove(k_pool + dst * blk, k_pool + src * blk, (size_t)blk);
    memmove(v_pool + dst * blk, v_pool + src * blk, (size_t)blk);
    if (kv_dtype == OR_E4M3_BLK) { /* a block's scales travel with its codes */
      long long tiles = tiles_bytes(kv_dtype, num_blocks, n_kv_heads, block_size, head_dim);
      for (int h = 0; h < n_kv_heads; ++h) {
        tile_scale_set(k_pool, tiles, n_kv_heads, dst, h, tile_scale_get(k_pool, tiles, n_kv_heads, src, h));
        tile_scale_set(v_pool, tiles, n_kv_heads, dst, h, tile_scale_get(v_pool, tiles, n_kv_heads, src, h));
      }
    }
  }
  return status;
}

/* ---------------------------------------------------------------------------
 * Textbook softmax attention of one query vector q[head_dim] over n keys and
 * values (row r of K at K + r*ld, of V at V + r*ld), all fp64.
 * Writes out[head_dim] and, if probs != NULL, probs[n].
 * ------------------------------------------------------------------------- */
static void attend(const double* q, const double* K, const double* V, long long ld, int n,
                   int head_dim, double softmax_scale, double* out, double* probs) {
  for (int i = 0; i < head_dim; ++i) out[i] = 0.0;
  if (n == 0) return;
  double* z = (double*)malloc(sizeof(double) * (size_t)n);
  double zmax = -INFINITY;
  for (int r = 0; r < n; ++r) {
    double dot = 0.0;
    for (int i = 0; i < head_dim; ++i) dot += q[i] * K[r * ld + i];
    z[r] = softmax_scale * dot;
    if (z[r] > zmax) zmax = z[r];
  }
  double sum = 0.0;
  for (int r = 0; r < n; ++r) {
    z[r] = exp(z[r] - zmax);
    sum += z[r];
  }
  for (int r = 0; r < n; ++r) {
    double p = z[r] / sum;
    if (probs) probs[r] = p;
    for (int i = 0; i < head_dim; ++i) out[i] += p * V[r * ld + i];
  }
  free(z);
}

/* ---------------------------------------------------------------------------
 * Paged decode attention.
 *   q            : [S][n_q_heads][head_dim] 16-bit bit patterns (q_dtype)
 *   block_tables : [S][max_blocks_per_seq] physical block ids
 *   ctx_lens     : [S] context length of each sequence (tokens)
 *   out          : [S][n_q_heads][head_dim] fp64
 *   probs        : optional [S][n_q_heads][max_ctx] fp64 (max_ctx = the
 *                  largest ctx_lens entry), softmax probabilities; NULL to skip
 * Returns 0, -1 on an invalid block id or context length (that sequence's
 * output is then left zero), -2 if n_q_heads is not a multiple of n_kv_heads.
 * ------------------------------------------------------------------------- */
int or_paged_attention(int kv_dtype, int q_dtype, int num_blocks, int block_size, int n_kv_heads,
                       int head_dim, const uint8_t* k_pool, const uint8_t* v_pool,
                       float k_scale, float v_scale, const uint16_t* q, int n_q_heads,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* ctx_lens, int S, double softmax_scale, double* out,
                       double* probs) {
  if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -2;
  int G = n_q_heads / n_kv_heads;
  int status = 0;
  int max_ctx = 0;
  for (int s = 0; s < S; ++s)
    if (ctx_lens[s] > max_ctx) max_ctx = ctx_lens[s];
  double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
  for (int s = 0; s < S; ++s) {
    int n = ctx_lens[s];
    double* o_seq = out + (long long)s * n_q_heads * head_dim;
    for (long long i = 0; i < (long long)n_q_heads * head_dim; ++i) o_seq[i] = 0.0;
    int nblk = (n + block_size - 1) / block_size;
    if (n < 0 || nblk > max_blocks_per_seq) {
      status = -1;
      continue;
    }
    int bad = 0;
    for (int j = 0; j < nblk; ++j) {
      int b = block_tables[(long long)s * max_blocks_per_seq + j];
      if (b < 0 || b >= num_blocks) bad = 1;
    }
    if (bad) {
      status = -1;
      continue;
    }
    /* Step 1: gather the sequence's pages, in logical order, into contiguous
     * K[n][n_kv_heads][head_dim] and V[...] (dequantising FP8 codes). */
    long long row = (long long)n_kv_heads * head_dim;
    long long tiles = tiles_bytes(kv_dtype, num_blocks, n_kv_heads, block_size, head_dim);
    double* K = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n * row : 1));
    double* V = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n * row : 1));
    for (int tok = 0; tok < n; ++tok) {
      int j = tok / block_size, off = tok % block_size;
      int b = block_tables[(long long)s * max_blocks_per_seq + j];
      for (int h = 0; h < n_kv_heads; ++h) {
        float ks = k_scale, vs = v_scale;
        if (kv_dtype == OR_E4M3_BLK) { /* the tile's own scales */
          ks = tile_scale_get(k_pool, tiles, n_kv_heads, b, h);
          vs = tile_scale_get(v_pool, tiles, n_kv_heads, b, h);
        }
        for (int i = 0; i < head_dim; ++i) {
          long long idx = pool_index(b, h, off, i, n_kv_heads, block_size, head_dim);
          K[tok * row + h * head_dim + i] = pool_value(kv_dtype, k_pool, idx, ks);
          V[tok * row + h * head_dim + i] = pool_value(kv_dtype, v_pool, idx, vs);
        }
      }
    }
    /* Step 2: softmax attention per query head against its kv head. */
    for (int g = 0; g < n_q_heads; ++g) {
      int h = g / G;
      const uint16_t* qg = q + ((long long)s * n_q_heads + g) * head_dim;
      for (int i = 0; i < head_dim; ++i) qv[i] = or_value16(q_dtype, qg[i]);
      double* pr = probs ? probs + ((long long)s * n_q_heads + g) * max_ctx : NULL;
      attend(qv, K + h * head_dim, V + h * head_dim, row, n, head_dim, softmax_scale,
             o_seq + (long long)g * head_dim, pr);
    }
    free(K);
    free(V);
  }
  free(qv);
  return status;
}

/* ---------------------------------------------------------------------------
 * Attention over a contiguous slab: K, V are [S][max_ctx][n_kv_heads][head_dim]
 * fp64 values, sequence s using its first ctx_lens[s] rows.  No pages, no
 * tables: the layout that paging replaces.  q is fp64 [S][n_q_heads][head_dim].
 * ------------------------------------------------------------------------- */
int or_slab_attention(const double* K, const double* V, int max_ctx, int n_kv_heads, int head_dim,
                      const double* q, int n_q_heads, const int32_t* ctx_lens, int S,
                      double softmax_scale, double* out) {
  if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -2;
  int G = n_q_heads / n_kv_heads;
  long long row = (long long)n_kv_heads * head_dim;
  for (int s = 0; s < S; ++s) {
    const double* Ks = K + (long long)s * max_ctx * row;
    const double* Vs = V + (long long)s * max_ctx * row;
    for (int g = 0; g < n_q_heads; ++g) {
      int h = g / G;
      attend(q + ((long long)s * n_q_heads + g) * head_dim, Ks + h * head_dim, Vs + h * head_dim,
             row, ctx_lens[s], head_dim, softmax_scale,
             out + ((long long)s * n_q_heads + g) * head_dim, NULL);
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Chunked prefill over the paged cache.
 *   q        : [T][n_q_heads][head_dim] 16-bit bit patterns; the chunk of
 *              sequence s is rows q_start[s] .. q_start[s+1]-1
 *   ctx_lens : [S] tokens of sequence s in the cache, the chunk included
 *   out      : [T][n_q_heads][head_dim] fp64
 * Returns 0, -1 on an invalid block id / length, -2 on a bad head count.
 * ------------------------------------------------------------------------- */
int or_paged_prefill(int kv_dtype, int q_dtype, int num_blocks, int block_size, int n_kv_heads,
                     int head_dim, const uint8_t* k_pool, const uint8_t* v_pool, float k_scale,
                     float v_scale, const uint16_t* q, int n_q_heads, const int32_t* q_start,
                     const int32_t* block_tables, int max_blocks_per_seq, const int32_t* ctx_lens,
                     int S, double softmax_scale, double* out) {
  if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -2;
  int G = n_q_heads / n_kv_heads;
  int status = 0;
  double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
  for (int s = 0; s < S; ++s) {
    int n = ctx_lens[s];
    int C = q_start[s + 1] - q_start[s];
    for (long long r = q_start[s]; r < q_start[s + 1]; ++r)
      for (long long i = 0; i < (long long)n_q_heads * head_dim; ++i)
        out[r * n_q_heads * head_dim + i] = 0.0;
    int nblk = (n + block_size - 1) / block_size;
    if (n < 0 || C < 0 || C > n || nblk > max_blocks_per_seq) {
      status = -1;
      continue;
    }
    int bad = 0;
    for (int j = 0; j < nblk; ++j) {
      int b = block_tables[(long long)s * max_blocks_per_seq + j];
      if (b < 0 || b >= num_blocks) bad = 1;
    }
    if (bad) {
      status = -1;
      continue;
    }
    /* gather the sequence's pages in logical order (as for decode) */
    long long row = (long long)n_kv_heads * head_dim;
    long long tiles = tiles_bytes(kv_dtype, num_blocks, n_kv_heads, block_size, head_dim);
    double* K = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n * row : 1));
    double* V = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n * row : 1));
    for (int tok = 0; tok < n; ++tok) {
      int j = tok / block_size, off = tok % block_size;
      int b = block_tables[(long long)s * max_blocks_per_seq + j];
      for (int h = 0; h < n_kv_heads; ++h) {
        float ks = k_scale, vs = v_scale;
        if (kv_dtype == OR_E4M3_BLK) { /* the tile's own scales */
          ks = tile_scale_get(k_pool, tiles, n_kv_heads, b, h);
          vs = tile_scale_get(v_pool, tiles, n_kv_heads, b, h);
        }
        for (int i = 0; i < head_dim; ++i) {
          long long idx = pool_index(b, h, off, i, n_kv_heads, block_size, head_dim);
          K[tok * row + h * head_dim + i] = pool_value(kv_dtype, k_pool, idx, ks);
          V[tok * row + h * head_dim + i] = pool_value(kv_dtype, v_pool, idx, vs);
        }
      }
    }
    /* query j sees tokens [0, n - C + j] */
    for (int j = 0; j < C; ++j) {
      long long r = q_start[s] + j;
      int visible = n - C + j + 1;
      for (int g = 0; g < n_q_heads; ++g) {
        int h = g / G;
        const uint16_t* qg = q + (r * n_q_heads + g) * head_dim;
        for (int i = 0; i < head_dim; ++i) qv[i] = or_value16(q_dtype, qg[i]);
        attend(qv, K + h * head_dim, V + h * head_dim, row, visible, head_dim, softmax_scale,
               out + (r * n_q_heads + g) * head_dim, NULL);
      }
    }
    free(K);
    free(V);
  }
  free(qv);
  return status;
}

/* Bytes of one block's record in a one-layer swap buffer: its K tiles of every
 * kv head, then its V tiles; a block-scaled pool adds the block's K scales and
 * V scales (n_kv_heads fp32 each) and zero bytes up to a multiple of 16. */
long long or_swap_record_bytes(int kv_dtype, int block_size, int n_kv_heads, int head_dim) {
  long long codes = 2LL * n_kv_heads * block_size * head_dim * elem_bytes(kv_dtype);
  if (kv_dtype != OR_E4M3_BLK) return codes;
  long long scales = 2LL * n_kv_heads * 4;
  return codes + (scales + 15) / 16 * 16;
}

/* Swap buffer of one layer: one record per listed block (above), records
 * back to back.  Returns -1 if an id is out of range (its record in buf is
 * left as is). */
int or_swap_gather(int kv_dtype, int num_blocks, int block_size, int n_kv_heads, int head_dim,
                   const int32_t* ids, int n, const uint8_t* k_pool, const uint8_t* v_pool,
                   uint8_t* buf) {
  long long blk = (long long)n_kv_heads * block_size * head_dim * elem_bytes(kv_dtype);
  long long rec = or_swap_record_bytes(kv_dtype, block_size, n_kv_heads, head_dim);
  long long tiles = tiles_bytes(kv_dtype, num_blocks, n_kv_heads, block_size, head_dim);
  int status = 0;
  for (int i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= num_blocks) {
      status = -1;
      continue;
    }
    uint8_t* r = buf + i * rec;
    memcpy(r, k_pool + ids[i] * blk, (size_t)blk);
    memcpy(r + blk, v_pool + ids[i] * blk, (size_t)blk);
    if (kv_dtype == OR_E4M3_BLK) {
      memset(r + 2 * blk, 0, (size_t)(rec - 2 * blk));
      memcpy(r + 2 * blk, k_pool + tiles + 4LL * ids[i] * n_kv_heads, 4 * (size_t)n_kv_heads);
      memcpy(r + 2 * blk + 4LL * n_kv_heads, v_pool + tiles + 4LL * ids[i] * n_kv_heads,
             4 * (size_t)n_kv_heads);
    }
  }
  return status;
}
