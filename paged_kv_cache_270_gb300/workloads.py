"""Seeded synthetic workloads for paged KV-cache decode.

This module only draws inputs: shapes, context lengths, block tables, and the
16-bit query / key / value bit patterns.  It holds none of the method's
arithmetic, and both the CUDA path's tests and the CPU oracle read the inputs
it makes.

Every draw is seeded (seed = 1000 + workload index) and is reproducible chunk
by chunk: the keys and values of sequence s, tokens [256c, 256c+256), come from
their own numpy generator keyed by (seed, s, c, stream), so a sampled check can
regenerate one sequence without drawing the others.  Values are N(0, 1) drawn in
float32, optionally scaled by 8 on a seeded 1% of key elements ("outliers"), then
rounded to the storage dtype (round-to-nearest-even).

Workloads (shapes follow the model families the pages name: Llama-3.1 8B and
70B with grouped-query attention 4:1 and 8:1, head dim 128, 16-token blocks):

  tiny_fp16            4 seqs, ctx {17, 33, 64, 100}, Hq 4 / Hkv 2, d 64, fp16,
                       32-block pool, tables a seeded random permutation
  llama3_8b_bf16       64 seqs, ctx ~ U[512, 4096], Hq 32 / Hkv 8, d 128, bf16,
                       pool 1.25x the blocks needed, shuffled
  llama3_8b_fp8        as llama3_8b_bf16 (same contexts), FP8 E4M3 cache with
                       per-tensor scales amax/448 over the generated K and V,
                       1% of K elements x8, then decode steps that each append
                       one token per sequence
  llama3_70b_fp8_a     Hq 64 / Hkv 8, d 128, FP8: 4 seqs x 131072 tokens
  llama3_70b_fp8_b     same shapes: 256 seqs x 4096 tokens
  llama3_70b_fp8_prefill  70B shapes, FP8: 4 sequences, each prefilling a
                       2048-token chunk after 6144 cached tokens (one
                       8192-token packet of chunked prefill)
  prefix_share_bf16    Hq 32 / Hkv 8, d 128, bf16: 64 requests sharing a
                       2048-token prefix, each with a U[128, 1024] suffix
                       (tables come from the block allocator, not from here)
  llama3_8b_fp8_long_short  8B shapes, FP8: one 131072-token sequence among 127
                       of U[128, 1024] tokens (a batch whose lengths differ by
                       orders of magnitude)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK = 16
CHUNK = 256  # tokens per independently seeded draw

NAMES = ("tiny_fp16", "llama3_8b_bf16", "llama3_8b_fp8", "llama3_8b_fp8_long_short", "llama3_70b_fp8_a",
         "llama3_70b_fp8_b", "llama3_70b_fp8_prefill", "prefix_share_bf16")


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + rounding) >> 16).astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float32 value of 16-bit patterns (used for amax only)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view(np.float16).astype(np.float32)


@dataclass
class Workload:
    name: str
    index: int                 # workload index; seed = 1000 + index
    kv_dtype: str              # "fp16" | "bf16" | "fp8_e4m3" | "fp8_e4m3_block"
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ctx_lens: np.ndarray       # int32 [S], context length at the first decode step
    num_blocks: int
    block_tables: np.ndarray   # int32 [S, max_blocks]; entries past a sequence's use are 0
    spare_blocks: list = field(default_factory=list)  # free physical ids, in draw order
    outlier_frac: float = 0.0
    outlier_mult: float = 8.0
    steps: int = 1             # decode steps (each appends one token per sequence)
    block_size: int = BLOCK
    k_scale: float = 1.0
    v_scale: float = 1.0
    kv_seed: int | None = None
    chunk: int = 0             # prefill workloads: new tokens per sequence (the last ones)

    # ----------------------------------------------------------------- shapes
    @property
    def S(self) -> int:
        return int(self.ctx_lens.shape[0])

    @property
    def G(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def in_dtype(self) -> str:
        """dtype of q and of the K/V handed to the cache (FP8 caches take bf16)."""
        return "fp16" if self.kv_dtype == "fp16" else "bf16"

    @property
    def elem_bytes(self) -> int:
        return 1 if self.kv_dtype in ("fp8_e4m3", "fp8_e4m3_block") else 2

    @property
    def block_scaled(self) -> bool:
        """FP8 with a dynamic scale per (block, kv head) tile, for K and for V."""
        return self.kv_dtype == "fp8_e4m3_block"

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def seed(self) -> int:
        return 1000 + self.index

    # ------------------------------------------------------------------ draws
    def _cast(self, x: np.ndarray) -> np.ndarray:
        return f32_to_f16_bits(x) if self.in_dtype == "fp16" else f32_to_bf16_bits(x)

    def _chunk(self, s: int, c: int):
        seed = self.kv_seed if self.kv_seed is not None else self.seed
        shape = (CHUNK, self.n_kv_heads, self.head_dim)
        rk = np.random.default_rng([seed, 1, s, c])
        k = rk.standard_normal(shape, dtype=np.float32)
        if self.outlier_frac > 0:
            mask = rk.random(shape, dtype=np.float32) < self.outlier_frac
            k = np.where(mask, k * np.float32(self.outlier_mult), k)
        rv = np.random.default_rng([seed, 2, s, c])
        v = rv.standard_normal(shape, dtype=np.float32)
        return self._cast(k), self._cast(v)

    def kv_bits(self, s: int, lo: int, hi: int):
        """K and V bit patterns [hi-lo, Hkv, d] of tokens [lo, hi) of sequence s."""
        ks, vs = [], []
        for c in range(lo // CHUNK, (hi + CHUNK - 1) // CHUNK):
            k, v = self._chunk(s, c)
            a, b = max(lo, c * CHUNK) - c * CHUNK, min(hi, (c + 1) * CHUNK) - c * CHUNK
            ks.append(k[a:b])
            vs.append(v[a:b])
        if not ks:
            z = np.zeros((0, self.n_kv_heads, self.head_dim), np.uint16)
            return z, z.copy()
        return np.concatenate(ks), np.concatenate(vs)

    def q_bits(self, step: int = 0) -> np.ndarray:
        rq = np.random.default_rng([self.seed, 3, step])
        q = rq.standard_normal((self.S, self.n_q_heads, self.head_dim), dtype=np.float32)
        return self._cast(q)

    def prefill_q_bits(self) -> np.ndarray:
        """Queries of the chunks, packed [S * chunk, Hq, d] (sequence-major)."""
        rq = np.random.default_rng([self.seed, 6])
        q = rq.standard_normal((self.S * self.chunk, self.n_q_heads, self.head_dim),
                               dtype=np.float32)
        return self._cast(q)

    def prefill_flops(self) -> int:
        """QK and PV multiply-adds of the causal chunks: query j of a chunk ending
        at ctx sees ctx - chunk + j + 1 keys; 4 * head_dim flops per key per head."""
        keys = sum(int(n) * self.chunk - self.chunk * (self.chunk - 1) // 2
                   for n in self.ctx_lens)
        return 4 * self.head_dim * self.n_q_heads * keys

    def final_ctx(self) -> np.ndarray:
        """Context lengths after the last decode step."""
        return self.ctx_lens + (self.steps - 1)

    def compute_fp8_scales(self) -> None:
        """Static per-tensor scales fl32(amax / 448) over every K and V value the
        workload generates (all tokens of all decode steps)."""
        if self.kv_dtype != "fp8_e4m3":
            return
        ka = va = np.float32(0)
        for s, n in enumerate(self.final_ctx()):
            for lo in range(0, int(n), 8 * CHUNK):
                k, v = self.kv_bits(s, lo, min(int(n), lo + 8 * CHUNK))
                ka = max(ka, np.abs(bits_to_f32(k, self.in_dtype)).max(initial=0))
                va = max(va, np.abs(bits_to_f32(v, self.in_dtype)).max(initial=0))
        self.k_scale = float(np.float32(ka) / np.float32(448.0))
        self.v_scale = float(np.float32(va) / np.float32(448.0))

    # -------------------------------------------------------------- placement
    def slots(self, s: int, lo: int, hi: int) -> np.ndarray:
        """Physical slot of each token in [lo, hi) of sequence s via its table."""
        pos = np.arange(lo, hi, dtype=np.int64)
        blk = self.block_tables[s, pos // self.block_size].astype(np.int64)
        return blk * self.block_size + pos % self.block_size

    def kv_bytes(self, ctx=None) -> int:
        """Algorithmic K+V bytes one decode pass reads (block-scaled pools add the
        two fp32 scales of every (page, kv head) tile read)."""
        ctx = np.asarray(self.ctx_lens if ctx is None else ctx, dtype=np.int64)
        n = int(np.sum(ctx)) * 2 * self.n_kv_heads * self.head_dim * self.elem_bytes
        if self.block_scaled:
            n += int(np.sum(-(-ctx // self.block_size))) * self.n_kv_heads * 8
        return n


def _tables_from_permutation(rng, ctx, num_blocks, max_blocks):
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.zeros((len(ctx), max_blocks), np.int32)
    used = 0
    for s, n in enumerate(ctx):
        nb = -(-int(n) // BLOCK)
        tables[s, :nb] = perm[used:used + nb]
        used += nb
    return tables, [int(b) for b in perm[used:]]


def _paged(index, name, kv_dtype, hq, hkv, d, ctx, num_blocks=None, slack=1.0, steps=1,
           outlier_frac=0.0, max_blocks=None, kv_seed=None):
    rng = np.random.default_rng([1000 + index, 0])
    ctx = np.asarray(ctx, dtype=np.int32)
    need_final = -(-(ctx + steps - 1) // BLOCK)
    if num_blocks is None:
        num_blocks = int(math.ceil(slack * int(np.sum(-(-ctx // BLOCK)))))
        num_blocks = max(num_blocks, int(np.sum(need_final)))
    if max_blocks is None:
        max_blocks = int(need_final.max(initial=1))
    tables, spare = _tables_from_permutation(rng, ctx, num_blocks, max_blocks)
    return Workload(name=name, index=index, kv_dtype=kv_dtype, n_q_heads=hq, n_kv_heads=hkv,
                    head_dim=d, ctx_lens=ctx, num_blocks=num_blocks, block_tables=tables,
                    spare_blocks=spare, outlier_frac=outlier_frac, steps=steps,
                    kv_seed=kv_seed)


def llama8b_contexts(S: int = 64) -> np.ndarray:
    rng = np.random.default_rng([1001, 5])
    return rng.integers(512, 4096, size=S, endpoint=True).astype(np.int32)


def make(name: str, scale_down: int = 1, steps: int | None = None) -> Workload:
    """Build a named workload.  ``scale_down`` > 1 shrinks sequence counts and
    lengths (for quick parity runs) while keeping head shapes and dtypes."""
    sd = max(1, int(scale_down))
    if "_fp8_block" in name:
        # the FP8 workload of the same shapes and values, with dynamic per-block scales
        w = make(name.replace("_fp8_block", "_fp8"), scale_down, steps)
        w.name, w.kv_dtype, w.k_scale, w.v_scale = name, "fp8_e4m3_block", 1.0, 1.0
        return w
    if name == "tiny_fp16":
        return _paged(0, name, "fp16", 4, 2, 64, [17, 33, 64, 100], num_blocks=32)
    if name == "llama3_8b_bf16":
        ctx = llama8b_contexts(max(2, 64 // sd))
        if sd > 1:
            ctx = np.maximum(1, ctx // sd).astype(np.int32)
        return _paged(1, name, "bf16", 32, 8, 128, ctx, slack=1.25)
    if name == "llama3_8b_fp8":
        ctx = llama8b_contexts(max(2, 64 // sd))
        if sd > 1:
            ctx = np.maximum(1, ctx // sd).astype(np.int32)
        w = _paged(2, name, "fp8_e4m3", 32, 8, 128, ctx, slack=1.25,
                   steps=32 if steps is None else steps, outlier_frac=0.01)
        return w
    if name == "llama3_8b_fp8_long_short":
        rng = np.random.default_rng([1006, 5])
        ctx = np.concatenate([[131072 // sd], rng.integers(128, 1024, size=max(1, 127 // sd),
                                                           endpoint=True) // sd])
        return _paged(6, name, "fp8_e4m3", 32, 8, 128, np.maximum(1, ctx).astype(np.int32))
    if name == "llama3_70b_fp8_a":
        return _paged(3, name, "fp8_e4m3", 64, 8, 128, [131072 // sd] * 4)
    if name == "llama3_70b_fp8_b":
        return _paged(3, name, "fp8_e4m3", 64, 8, 128, [4096 // sd] * max(2, 256 // sd),
                      kv_seed=1003 + 10_000)
    if name == "llama3_70b_fp8_prefill":
        # one 8,192-token prefill packet: 4 sequences x 2,048 new tokens after 6,144 cached
        w = _paged(5, name, "fp8_e4m3", 64, 8, 128, [(6144 + 2048) // sd] * 4)
        w.chunk = 2048 // sd
        return w
    raise KeyError(name)


# ----------------------------------------------------------- prefix sharing
@dataclass
class PrefixShare:
    """Draws for the prefix-sharing / branching workload (index 4, bf16)."""
    n_requests: int = 64
    prefix_tokens: int = 2048
    suffix_lo: int = 128
    suffix_hi: int = 1024
    n_q_heads: int = 32
    n_kv_heads: int = 8
    head_dim: int = 128
    kv_dtype: str = "bf16"
    seed: int = 1004

    def suffix_lens(self) -> np.ndarray:
        rng = np.random.default_rng([self.seed, 0])
        return rng.integers(self.suffix_lo, self.suffix_hi, size=self.n_requests,
                            endpoint=True).astype(np.int32)

    def _draw(self, stream: int, key: int, n: int):
        shape = (n, self.n_kv_heads, self.head_dim)
        r = np.random.default_rng([self.seed, stream, key])
        return f32_to_bf16_bits(r.standard_normal(shape, dtype=np.float32))

    def prefix_kv(self, n: int | None = None):
        n = self.prefix_tokens if n is None else n
        return self._draw(1, 0, n), self._draw(2, 0, n)

    def suffix_kv(self, r: int, n: int):
        return self._draw(3, r + 1, n), self._draw(4, r + 1, n)

    def q_bits(self, S: int, step: int = 0) -> np.ndarray:
        rq = np.random.default_rng([self.seed, 5, step])
        return f32_to_bf16_bits(
            rq.standard_normal((S, self.n_q_heads, self.head_dim), dtype=np.float32))
