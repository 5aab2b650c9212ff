"""Seeded random cases of decode and chunked prefill against the fp64 oracle.
Each case draws the pool type, head dim, query heads per KV head (1 to 8, so
the tensor-core prefill and the mma.sync kernels both run), KV heads, batch,
ragged contexts (one token, page boundaries, several pages), split counts and
chunk lengths; every slot the tables do not reach holds 0xFF bytes (NaN in
16 bits, NaN codes in E4M3), and the block tables are a random permutation."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import (bits_to_torch, check_fp32, check_half, fill_both, gpu_decode, new_pool,
                         oracle_decode, oracle_pools, vmax_of)
from paged_kv_cache_270_gb300 import _native as N
from paged_kv_cache_270_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DTYPES = ["fp16", "bf16", "fp8_e4m3", "fp8_e4m3_block"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_270_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    oracle.build()


def _case(seed):
    rng = np.random.default_rng([seed, 2027])
    kv_dtype = DTYPES[seed % len(DTYPES)]
    d = int(rng.choice([64, 128]))
    G = int(rng.integers(1, 9))
    Hkv = int(rng.integers(1, 4))
    S = int(rng.integers(1, 7))
    # contexts: a mix of one token, exact page multiples and its neighbours, and random lengths
    pool_of = [1, 15, 16, 17, 31, 32, 33, 127, 128, 129, 255, 256, 257]
    ctx = np.array([int(rng.choice(pool_of)) if rng.random() < 0.5 else int(rng.integers(1, 700))
                    for _ in range(S)], np.int32)
    max_blocks = int(-(-int(ctx.max()) // 16)) + int(rng.integers(0, 3))
    nb = int(np.sum(-(-ctx // 16))) + int(rng.integers(1, 6))
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.zeros((S, max_blocks), np.int32)
    used = 0
    for s, n in enumerate(ctx):
        k = -(-int(n) // 16)
        tables[s, :k] = perm[used:used + k]
        tables[s, k:] = rng.integers(-7, 10**6, max_blocks - k)  # never read
        used += k
    w = W.Workload(name=f"fuzz{seed}", index=20 + seed, kv_dtype=kv_dtype, n_q_heads=Hkv * G,
                   n_kv_heads=Hkv, head_dim=d, ctx_lens=ctx, num_blocks=nb, block_tables=tables,
                   kv_seed=seed)
    w.compute_fp8_scales()
    return w, rng


@pytest.mark.parametrize("seed", range(16))
def test_random_decode(seed):
    w, rng = _case(seed)
    pool = new_pool(w, 0xFF)
    op = oracle_pools(w, 0xFF)
    fill_both(w, pool, op)
    q = w.q_bits()
    ref = oracle_decode(w, op, q)
    vmax = vmax_of(w, op)
    for ns in (0, 1, int(rng.integers(2, 40))):
        check_half(gpu_decode(w, pool, q, num_splits=ns), ref, vmax)
        check_fp32(gpu_decode(w, pool, q, out_dtype=torch.float32, num_splits=ns), ref)
    assert pool.device_error() == N.PA_OK


@pytest.mark.parametrize("seed", range(16))
def test_random_prefill(seed):
    w, rng = _case(seed)
    pool = new_pool(w, 0xFF)
    op = oracle_pools(w, 0xFF)
    fill_both(w, pool, op)
    # each sequence's last c tokens are its chunk (1 <= c <= ctx)
    chunks = np.array([int(rng.integers(1, int(n) + 1)) for n in w.ctx_lens], np.int32)
    T = int(chunks.sum())
    x = rng.standard_normal((T, w.n_q_heads, w.head_dim), dtype=np.float32)
    q = W.f32_to_f16_bits(x) if w.in_dtype == "fp16" else W.f32_to_bf16_bits(x)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    ref = oracle.paged_prefill(w.kv_dtype, w.in_dtype, w.num_blocks, 16, w.n_kv_heads, w.head_dim,
                               op[0], op[1], w.k_scale, w.v_scale, q, q_start, w.block_tables,
                               w.ctx_lens, w.softmax_scale)
    args = (bits_to_torch(q, w.in_dtype), torch.from_numpy(q_start).cuda(),
            torch.from_numpy(w.block_tables).cuda(), torch.from_numpy(w.ctx_lens).cuda())
    mc = int(chunks.max())
    check_half(pool.prefill(*args, max_chunk=mc, softmax_scale=w.softmax_scale), ref, vmax_of(w, op))
    check_fp32(pool.prefill(*args, max_chunk=mc, softmax_scale=w.softmax_scale, out_dtype=torch.float32),
               ref)
    torch.cuda.synchronize()
    assert pool.device_error() == N.PA_OK
