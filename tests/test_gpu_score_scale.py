"""Score scales away from the usual 1/sqrt(head_dim), against the fp64 oracle:
zero (every visible key weighs the same, so an output row is the mean of its
visible V rows) and negative (the softmax of the negated scores).  Decode,
the mma.sync prefill (head_dim 64) and the tensor-core prefill (head_dim 128)
all run, with causal diagonals, so masked keys meet the zero factor."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import bits_to_torch, check_fp32, check_half, fill_both, new_pool, oracle_pools, vmax_of
from paged_kv_cache_270_gb300 import _native as N
from paged_kv_cache_270_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SCALES = [0.0, -0.0625]
KINDS = ["fp8_e4m3", "fp8_e4m3_block", "bf16", "fp16"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_270_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    oracle.build()


def _workload(kv_dtype, d, G, ctx, seed, Hkv=2):
    ctx = np.asarray(ctx, np.int32)
    max_blocks = int(-(-int(ctx.max()) // 16))
    nb = int(np.sum(-(-ctx // 16))) + 2
    rng = np.random.default_rng(seed)
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.zeros((len(ctx), max_blocks), np.int32)
    used = 0
    for s, n in enumerate(ctx):
        k = -(-int(n) // 16)
        tables[s, :k] = perm[used:used + k]
        tables[s, k:] = rng.integers(-3, 10**6, max_blocks - k)  # never read
        used += k
    w = W.Workload(name=f"scale_{kv_dtype}_{d}", index=9, kv_dtype=kv_dtype, n_q_heads=G * Hkv,
                   n_kv_heads=Hkv, head_dim=d, ctx_lens=ctx, num_blocks=nb, block_tables=tables,
                   kv_seed=seed)
    w.compute_fp8_scales()
    return w


def _queries(w, T, seed):
    x = np.random.default_rng([seed, 5]).standard_normal((T, w.n_q_heads, w.head_dim),
                                                         dtype=np.float32)
    return W.f32_to_f16_bits(x) if w.in_dtype == "fp16" else W.f32_to_bf16_bits(x)


def _check(w, op, out, out32, ref):
    check_half(out, ref, vmax_of(w, op))
    check_fp32(out32, ref)


@pytest.mark.parametrize("kv_dtype", KINDS)
@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("num_splits", [0, 3])
def test_decode(kv_dtype, scale, num_splits):
    ctx = [1, 17, 300, 1000]
    w = _workload(kv_dtype, 128, 8, ctx, seed=61)
    pool, op = new_pool(w, 0xFF), oracle_pools(w, 0xFF)
    fill_both(w, pool, op)
    q = _queries(w, len(ctx), seed=62)
    ref = oracle.paged_attention(w.kv_dtype, w.in_dtype, w.num_blocks, 16, w.n_kv_heads, 128,
                                 op[0], op[1], w.k_scale, w.v_scale, q, w.block_tables,
                                 w.ctx_lens, scale)
    args = (bits_to_torch(q, w.in_dtype), torch.from_numpy(w.block_tables).cuda(),
            torch.from_numpy(w.ctx_lens).cuda())
    out = pool.decode(*args, softmax_scale=scale, num_splits=num_splits)
    out32 = pool.decode(*args, softmax_scale=scale, num_splits=num_splits,
                        out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pool.device_error() == N.PA_OK
    _check(w, op, out, out32, ref)


@pytest.mark.parametrize("kv_dtype", KINDS)
@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("d", [64, 128])
def test_prefill(kv_dtype, scale, d):
    # (history, chunk): diagonals inside a page, across 128-key blocks, one-token chunks
    pairs = [(0, 1), (0, 40), (150, 130), (700, 64), (33, 1)]
    ctx = [h + c for h, c in pairs]
    chunks = [c for _, c in pairs]
    w = _workload(kv_dtype, d, 8, ctx, seed=63 + d)
    pool, op = new_pool(w, 0xFF), oracle_pools(w, 0xFF)
    fill_both(w, pool, op)
    q = _queries(w, sum(chunks), seed=64)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    ref = oracle.paged_prefill(w.kv_dtype, w.in_dtype, w.num_blocks, 16, w.n_kv_heads, d, op[0],
                               op[1], w.k_scale, w.v_scale, q, q_start, w.block_tables,
                               w.ctx_lens, scale)
    args = (bits_to_torch(q, w.in_dtype), torch.from_numpy(q_start).cuda(),
            torch.from_numpy(w.block_tables).cuda(), torch.from_numpy(w.ctx_lens).cuda())
    out = pool.prefill(*args, max_chunk=max(chunks), softmax_scale=scale)
    out32 = pool.prefill(*args, max_chunk=max(chunks), softmax_scale=scale,
                         out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pool.device_error() == N.PA_OK
    _check(w, op, out, out32, ref)
