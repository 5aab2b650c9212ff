"""GPU parity of the tensor-core (tcgen05) chunked prefill against the fp64
oracle.  pa_prefill takes that path for pools with head_dim 128 and 8 query
heads per KV head (1, 2, 4 or 8; FP8 static or block-scaled, bfloat16, binary16); these cases
make it run many 128-key blocks (the ring
wraps many times), ragged query tiles, causal diagonals at every offset,
both FP8 scalings and both output types, and scores that grow block after
block so the running max moves by more than 2^8 and O is rescaled in tensor
memory."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import bits_to_torch, check_fp32, check_half, new_pool, oracle_pools, vmax_of
from paged_kv_cache_270_gb300 import _native as N
from paged_kv_cache_270_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_270_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    oracle.build()


def _setup(kv_dtype, pairs, seed, Hkv=2, k_gain_per_block=1.0, q_away_from_zero=False, G=8):
    ctx = np.array([h + c for h, c in pairs], np.int32)
    chunks = [c for _, c in pairs]
    max_blocks = int(-(-ctx.max() // 16))
    nb = int(np.sum(-(-ctx // 16))) + 2
    rng = np.random.default_rng(seed)
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.zeros((len(ctx), max_blocks), np.int32)
    used = 0
    for s, n in enumerate(ctx):
        k = -(-int(n) // 16)
        tables[s, :k] = perm[used:used + k]
        tables[s, k:] = rng.integers(-5, 10**6, max_blocks - k)  # never read
        used += k
    w = W.Workload(name="tc", index=12, kv_dtype=kv_dtype, n_q_heads=G * Hkv, n_kv_heads=Hkv,
                   head_dim=128, ctx_lens=ctx, num_blocks=nb, block_tables=tables, kv_seed=seed)
    # K/V values: N(0,1); optionally K grows by a factor per 128-token block
    kv = []
    for s, n in enumerate(ctx):
        k, v = w.kv_bits(s, 0, int(n))
        if k_gain_per_block != 1.0:
            g = np.power(k_gain_per_block, np.arange(int(n)) // 128).astype(np.float32)
            k = _cast(w, W.bits_to_f32(k, w.in_dtype) * g[:, None, None])
        kv.append((k, v))
    if kv_dtype == "fp8_e4m3":
        ka = max(float(np.abs(W.bits_to_f32(k, w.in_dtype)).max()) for k, _ in kv)
        va = max(float(np.abs(W.bits_to_f32(v, w.in_dtype)).max()) for _, v in kv)
        w.k_scale = float(np.float32(ka) / np.float32(448))
        w.v_scale = float(np.float32(va) / np.float32(448))
    pool = new_pool(w, 0xFF)
    op = oracle_pools(w, 0xFF)
    for s, (k, v) in enumerate(kv):
        slots = w.slots(s, 0, int(ctx[s]))
        pool.reshape_and_cache(bits_to_torch(k, w.in_dtype), bits_to_torch(v, w.in_dtype),
                               torch.from_numpy(slots).cuda())
        assert oracle.reshape_and_cache(kv_dtype, nb, 16, Hkv, 128, k, v, slots, w.k_scale,
                                        w.v_scale, *op) == 0
    T = sum(chunks)
    qf = rng.standard_normal((T, G * Hkv, 128)).astype(np.float32)
    if q_away_from_zero:  # |q| in [0.5, 2): the two-term E4M3 split of q is exact
        qf = (np.sign(qf) * rng.uniform(0.5, 2.0, qf.shape)).astype(np.float32)
    q = _cast(w, qf)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    return w, pool, op, q, q_start, chunks


def _cast(w, x):
    return W.f32_to_f16_bits(x) if w.in_dtype == "fp16" else W.f32_to_bf16_bits(x)


def _run(w, pool, op, q, q_start, chunks):
    ref = oracle.paged_prefill(w.kv_dtype, w.in_dtype, w.num_blocks, 16, w.n_kv_heads, 128, op[0],
                               op[1], w.k_scale, w.v_scale, q, q_start, w.block_tables, w.ctx_lens,
                               w.softmax_scale)
    args = (bits_to_torch(q, w.in_dtype), torch.from_numpy(q_start).cuda(),
            torch.from_numpy(w.block_tables).cuda(), torch.from_numpy(w.ctx_lens).cuda())
    out = pool.prefill(*args, max_chunk=max(chunks), softmax_scale=w.softmax_scale)
    out32 = pool.prefill(*args, max_chunk=max(chunks), softmax_scale=w.softmax_scale,
                         out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pool.device_error() == N.PA_OK
    check_half(out, ref, vmax_of(w, op))
    check_fp32(out32, ref)
    return out32, ref


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "fp8_e4m3_block", "bf16", "fp16"])
def test_long_histories_ragged_tiles(kv_dtype):
    # (history, chunk): 1-token chunks, chunks ending inside a page, a chunk
    # whose diagonal crosses a 128-key block, 3000 keys of history (24 blocks)
    pairs = [(0, 1), (0, 16), (3000, 20), (700, 200), (0, 300), (129, 1), (250, 64), (127, 129)]
    w, pool, op, q, q_start, chunks = _setup(kv_dtype, pairs, seed=41)
    _run(w, pool, op, q, q_start, chunks)


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "fp8_e4m3_block", "bf16", "fp16"])
def test_scores_growing_block_after_block(kv_dtype):
    """K doubles every 128 tokens: each block's scores exceed the previous
    max by far more than 2^8 in the exponent, so every block rescales O.
    Logits reach hundreds of log2 units here, which would magnify the query
    split's rounding (elements below ~2^-9 of the row max); q is drawn away
    from zero so the split is exact and the test isolates the rescaling."""
    pairs = [(900, 100), (500, 33)]
    w, pool, op, q, q_start, chunks = _setup(kv_dtype, pairs, seed=43, k_gain_per_block=2.0,
                                             q_away_from_zero=True)
    _run(w, pool, op, q, q_start, chunks)


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "fp8_e4m3_block", "bf16"])
@pytest.mark.parametrize("G", [1, 2, 4])
def test_fewer_heads_per_group_longer_tiles(kv_dtype, G):
    """G query heads per KV head: a tile is 128 / G tokens (128 for G = 1), so
    chunks span several tiles with a ragged last one and diagonals cross
    128-key blocks at every offset."""
    pairs = [(0, 1), (3000, 200), (129, 130), (700, 64), (0, 257)]
    w, pool, op, q, q_start, chunks = _setup(kv_dtype, pairs, seed=53 + G, G=G)
    _run(w, pool, op, q, q_start, chunks)


def test_many_heads_and_sequences_match_mma_sync_shapes():
    """Hkv 8 (64 query heads), 6 sequences: every (tile, kv head, sequence) CTA."""
    pairs = [(0, 48), (17, 31), (256, 256), (1000, 5), (64, 64), (0, 129)]
    w, pool, op, q, q_start, chunks = _setup("fp8_e4m3", pairs, seed=47, Hkv=8)
    _run(w, pool, op, q, q_start, chunks)


def test_bounds_still_reported():
    pairs = [(40, 10)]
    w, pool, op, q, q_start, chunks = _setup("fp8_e4m3", pairs, seed=49)
    bad = w.block_tables.copy()
    bad[0, 1] = w.num_blocks + 7
    pool.prefill(bits_to_torch(q, "bf16"), torch.from_numpy(q_start).cuda(),
                 torch.from_numpy(bad).cuda(), torch.from_numpy(w.ctx_lens).cuda(), max_chunk=10)
    assert pool.device_error() == N.PA_ERR_BOUNDS
    long_chunk = np.array([0, 60], np.int32)  # longer than the context
    qq = W.f32_to_bf16_bits(np.zeros((60, 16, 128), np.float32))
    pool.prefill(bits_to_torch(qq, "bf16"), torch.from_numpy(long_chunk).cuda(),
                 torch.from_numpy(w.block_tables).cuda(), torch.from_numpy(w.ctx_lens).cuda(),
                 max_chunk=60)
    assert pool.device_error() == N.PA_ERR_BOUNDS
    # a chunk longer than the grid max_chunk sizes (one tile of 128 / G = 16
    # rows here): those rows are written, the rest are not, and the error is reported
    args = (torch.from_numpy(w.block_tables).cuda(), torch.from_numpy(w.ctx_lens).cuda())
    q40 = W.f32_to_bf16_bits(np.ones((40, 16, 128), np.float32))
    out = torch.full((40, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    pool.prefill(bits_to_torch(q40, "bf16"), torch.tensor([0, 40], dtype=torch.int32, device="cuda"),
                 *args, max_chunk=10, out=out)
    assert pool.device_error() == N.PA_ERR_BOUNDS
    assert torch.isfinite(out[:16]).all() and torch.isnan(out[16:]).all()
    # a negative start and a decreasing pair: the sequence is skipped
    for bad_start in ([-4, 10], [10, 4]):
        pool.prefill(bits_to_torch(q40, "bf16"), torch.tensor(bad_start, dtype=torch.int32, device="cuda"),
                     *args, max_chunk=16, out=out)
        assert pool.device_error() == N.PA_ERR_BOUNDS
    _run(w, pool, op, q, q_start, chunks)


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "bf16"])
def test_back_to_back_launches_identical_and_error_free(kv_dtype):
    """Thirty launches in a row on one stream, the first right after the pool
    is filled (cold caches): each is bit-identical to the first and none
    records an error.  A barrier awaited by parity that fell two phases
    behind its producer would show as a wait running out its limit
    (PA_ERR_TIMEOUT); a race on a buffer, as a different result.  The first
    launch is also checked against the oracle."""
    pairs = [(2000, 300), (500, 128), (0, 77), (3000, 16)]
    w, pool, op, q, q_start, chunks = _setup(kv_dtype, pairs, seed=61)
    args = (bits_to_torch(q, w.in_dtype), torch.from_numpy(q_start).cuda(),
            torch.from_numpy(w.block_tables).cuda(), torch.from_numpy(w.ctx_lens).cuda())
    first = pool.prefill(*args, max_chunk=max(chunks), softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    assert pool.device_error() == N.PA_OK
    ref = oracle.paged_prefill(w.kv_dtype, w.in_dtype, w.num_blocks, 16, w.n_kv_heads, 128, op[0],
                               op[1], w.k_scale, w.v_scale, q, q_start, w.block_tables, w.ctx_lens,
                               w.softmax_scale)
    check_half(first, ref, vmax_of(w, op))
    outs = [pool.prefill(*args, max_chunk=max(chunks), softmax_scale=w.softmax_scale)
            for _ in range(30)]
    torch.cuda.synchronize()
    assert pool.device_error() == N.PA_OK
    for i, out in enumerate(outs):
        assert torch.equal(out.view(torch.int16), first.view(torch.int16)), f"launch {i + 1} differs"
