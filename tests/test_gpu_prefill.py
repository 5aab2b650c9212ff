"""GPU parity of pa_prefill (chunked prefill) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_harness import (FP32_ROW_TOL, bits_to_torch, check_fp32, check_half, fill_both, gpu_decode,
                         new_pool, oracle_decode, oracle_pools, vmax_of)
from paged_kv_cache_270_gb300 import _native as N
from paged_kv_cache_270_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_270_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    oracle.build()


def _workload(kv_dtype, d, G, ctx, seed, Hkv=2):
    ctx = np.asarray(ctx, np.int32)
    max_blocks = int(max(1, -(-int(ctx.max()) // 16)))
    nb = int(np.sum(-(-ctx // 16))) + 3
    rng = np.random.default_rng(seed)
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.zeros((len(ctx), max_blocks), np.int32)
    used = 0
    for s, n in enumerate(ctx):
        k = -(-int(n) // 16)
        tables[s, :k] = perm[used:used + k]
        tables[s, k:] = rng.integers(-3, 10**6, max_blocks - k)  # never read
        used += k
    w = W.Workload(name=f"prefill_{kv_dtype}_{d}_{G}", index=8, kv_dtype=kv_dtype,
                   n_q_heads=Hkv * G, n_kv_heads=Hkv, head_dim=d, ctx_lens=ctx, num_blocks=nb,
                   block_tables=tables)
    w.compute_fp8_scales()
    return w


def _chunk_queries(w, chunks, seed):
    rng = np.random.default_rng([seed, 77])
    T = int(sum(chunks))
    x = rng.standard_normal((T, w.n_q_heads, w.head_dim), dtype=np.float32)
    q = W.f32_to_f16_bits(x) if w.in_dtype == "fp16" else W.f32_to_bf16_bits(x)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    return q, q_start


def _gpu_prefill(w, pool, q_bits, q_start, out_dtype=None, ctx=None, tables=None):
    q = bits_to_torch(q_bits, w.in_dtype)
    qs = torch.from_numpy(q_start).cuda()
    t = torch.from_numpy(np.ascontiguousarray(w.block_tables if tables is None else tables)).cuda()
    c = torch.from_numpy(np.ascontiguousarray(w.ctx_lens if ctx is None else ctx)).cuda()
    chunks = np.diff(q_start)
    out = pool.prefill(q, qs, t, c, max_chunk=int(chunks.max(initial=0)), out_dtype=out_dtype,
                       softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    return out


def _oracle_prefill(w, op, q_bits, q_start):
    return oracle.paged_prefill(w.kv_dtype, w.in_dtype, w.num_blocks, 16, w.n_kv_heads,
                                w.head_dim, op[0], op[1], w.k_scale, w.v_scale, q_bits, q_start,
                                w.block_tables, w.ctx_lens, w.softmax_scale)


@pytest.mark.parametrize("kv_dtype", ["fp16", "bf16", "fp8_e4m3"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_prefill_shapes_and_ragged_chunks(kv_dtype, d, G):
    # (history before the chunk, chunk length) per sequence
    pairs = [(0, 1), (0, 17), (5, 16), (30, 33), (100, 100), (200, 3), (16, 16), (0, 64)]
    ctx = [h + c for h, c in pairs]
    chunks = [c for _, c in pairs]
    w = _workload(kv_dtype, d, G, ctx, seed=G * 100 + d)
    pool = new_pool(w, 0xFF)
    op = oracle_pools(w, 0xFF)
    fill_both(w, pool, op)
    q, q_start = _chunk_queries(w, chunks, seed=G + d)
    ref = _oracle_prefill(w, op, q, q_start)
    vmax = vmax_of(w, op)
    check_half(_gpu_prefill(w, pool, q, q_start), ref, vmax)
    check_fp32(_gpu_prefill(w, pool, q, q_start, out_dtype=torch.float32), ref)
    assert pool.device_error() == N.PA_OK


def test_one_token_chunks_match_decode():
    """A chunk of one token is a decode: both calls meet the fp32-mode bound
    against the oracle's decode, so they agree per row within twice it.  (The
    two kernels differ in how they carry P -- at these shapes the prefill runs
    on the tensor-core kernel, whose running max moves in steps of 2^8 -- so
    they are not compared element by element at a tighter tolerance.)"""
    w = W.make("llama3_8b_bf16", scale_down=8)
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    fill_both(w, pool, op)
    q_bits = w.q_bits()
    ref = oracle_decode(w, op, q_bits)
    q_start = np.arange(w.S + 1, dtype=np.int32)
    pre = _gpu_prefill(w, pool, q_bits.reshape(w.S, w.n_q_heads, w.head_dim), q_start,
                       out_dtype=torch.float32)
    dec = gpu_decode(w, pool, q_bits, out_dtype=torch.float32)
    check_fp32(pre, ref)
    check_fp32(dec, ref)
    diff = (pre - dec).abs().amax(dim=-1).double().cpu().numpy()
    scale = np.abs(ref).max(axis=-1)
    assert np.all(diff <= 2 * FP32_ROW_TOL * scale + 1e-30)


def test_prefill_in_two_chunks_matches_one_chunk():
    """Chunks interleaved with other work give the rows a single chunk gives."""
    w = _workload("bf16", 128, 4, [300], seed=5, Hkv=8)
    pool = new_pool(w, 0)
    fill_both(w, pool, None)
    q, _ = _chunk_queries(w, [300], seed=9)
    one = _gpu_prefill(w, pool, q, np.array([0, 300], np.int32), out_dtype=torch.float32)
    first = _gpu_prefill(w, pool, q[:123], np.array([0, 123], np.int32), out_dtype=torch.float32,
                         ctx=np.array([123], np.int32))
    second = _gpu_prefill(w, pool, q[123:], np.array([0, 177], np.int32), out_dtype=torch.float32)
    both = torch.cat([first, second])
    assert torch.allclose(one, both, rtol=1e-5, atol=1e-6)


@pytest.mark.slow
def test_prefill_70b_fp8_8192_token_packet_sampled():
    """Four sequences each prefilling a 2048-token chunk after 6144 cached tokens
    (one 8,192-token packet), 70B shapes, FP8: cache and sampled rows vs oracle."""
    S, hist, C = 4, 6144, 2048
    ctx = np.full(S, hist + C, np.int32)
    nb = S * (hist + C) // 16
    perm = np.random.default_rng(31).permutation(nb).astype(np.int32)
    w = W.Workload(name="prefill70b", index=9, kv_dtype="fp8_e4m3", n_q_heads=64, n_kv_heads=8,
                   head_dim=128, ctx_lens=ctx, num_blocks=nb,
                   block_tables=perm.reshape(S, -1).copy())
    w.compute_fp8_scales()
    pool = new_pool(w, None)
    fill_both(w, pool, None, chunk_tokens=1 << 15)
    q, q_start = _chunk_queries(w, [C] * S, seed=3)
    out = _gpu_prefill(w, pool, q, q_start)
    out32 = _gpu_prefill(w, pool, q, q_start, out_dtype=torch.float32)
    assert pool.device_error() == N.PA_OK
    # sample rows: each is a decode at its own position over the same pages
    rng = np.random.default_rng(4)
    rows = [(s, int(j)) for s in range(S) for j in rng.choice(C, 3, replace=False)] + [(0, 0), (3, C - 1)]
    for s in sorted(set(r for r, _ in rows)):
        ids = w.block_tables[s]
        ow = W.Workload(**{**w.__dict__, "ctx_lens": ctx[s:s + 1],
                           "block_tables": np.arange(len(ids), dtype=np.int32)[None, :],
                           "num_blocks": len(ids)})
        op = oracle_pools(ow, 0)
        n = int(ctx[s])
        for lo in range(0, n, 1 << 15):
            hi = min(n, lo + (1 << 15))
            k, v = w.kv_bits(s, lo, hi)
            pos = np.arange(lo, hi, dtype=np.int64)
            slots = pos  # compact pool: sequence s occupies blocks 0.. in order
            oracle.reshape_and_cache("fp8_e4m3", len(ids), 16, 8, 128, k, v, slots, w.k_scale,
                                     w.v_scale, *op)
        for (ss, j) in rows:
            if ss != s:
                continue
            r = q_start[s] + j
            ref = oracle.paged_attention("fp8_e4m3", "bf16", len(ids), 16, 8, 128, op[0], op[1],
                                         w.k_scale, w.v_scale, q[r:r + 1], ow.block_tables,
                                         np.array([hist + j + 1], np.int32), w.softmax_scale)
            check_half(out[r:r + 1], ref, vmax_of(ow, op))
            check_fp32(out32[r:r + 1], ref)


def test_prefill_bounds_reported():
    w = _workload("fp16", 64, 2, [40], seed=1)
    pool = new_pool(w, 0)
    fill_both(w, pool, None)
    q, q_start = _chunk_queries(w, [50], seed=2)      # chunk longer than the context
    _gpu_prefill(w, pool, q, q_start)
    assert pool.device_error() == N.PA_ERR_BOUNDS
    q, q_start = _chunk_queries(w, [10], seed=2)
    bad = w.block_tables.copy()
    bad[0, 1] = w.num_blocks + 5
    _gpu_prefill(w, pool, q, q_start, tables=bad)
    assert pool.device_error() == N.PA_ERR_BOUNDS
    _gpu_prefill(w, pool, q, q_start)
    assert pool.device_error() == N.PA_OK
    t = torch.from_numpy(w.block_tables).cuda()
    c = torch.from_numpy(w.ctx_lens).cuda()
    q40, qs40 = _chunk_queries(w, [40], seed=3)
    # a chunk longer than the grid max_chunk sizes: the rows the grid covers
    # are written, the rest are not, and the error is reported
    out = torch.full((40, w.n_q_heads, w.head_dim), float("nan"), dtype=torch.float16, device="cuda")
    pool.prefill(bits_to_torch(q40, "fp16"), torch.from_numpy(qs40).cuda(), t, c, max_chunk=16,
                 out=out)
    assert pool.device_error() == N.PA_ERR_BOUNDS
    assert torch.isfinite(out[:16]).all() and torch.isnan(out[16:]).all()
    # a negative start and a decreasing pair: the sequence is skipped
    for bad_start in ([-4, 10], [10, 4]):
        pool.prefill(bits_to_torch(q40, "fp16"), torch.tensor(bad_start, dtype=torch.int32,
                                                               device="cuda"),
                     t, c, max_chunk=16, out=out)
        assert pool.device_error() == N.PA_ERR_BOUNDS
    _gpu_prefill(w, pool, q, q_start)
    assert pool.device_error() == N.PA_OK
