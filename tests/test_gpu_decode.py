"""GPU parity of pa_decode against the fp64 oracle on every workload, plus the
method's invariances and degenerate cases, all through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_harness import (bits_to_torch, check_fp32, check_half, fill_both, full_size_sampled_check,
                         gpu_decode, new_pool, oracle_decode, oracle_pools, pool_bytes_equal,
                         vmax_of)
from paged_kv_cache_270_gb300 import _native as N
from paged_kv_cache_270_gb300 import workloads as W
from paged_kv_cache_270_gb300.pool import KVPool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_270_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    oracle.build()


def _run_full(w, splits_list=(0,), fill=0x00):
    w.compute_fp8_scales()
    pool = new_pool(w, fill)
    op = oracle_pools(w, fill)
    fill_both(w, pool, op)
    q = w.q_bits()
    ref = oracle_decode(w, op, q)
    vmax = vmax_of(w, op)
    for ns in splits_list:
        out = gpu_decode(w, pool, q, num_splits=ns)
        check_half(out, ref, vmax)
        out32 = gpu_decode(w, pool, q, out_dtype=torch.float32, num_splits=ns)
        check_fp32(out32, ref)
    assert pool.device_error() == N.PA_OK
    return pool, op, q, ref


def test_tiny_fp16_all_split_counts():
    w = W.make("tiny_fp16")
    _run_full(w, splits_list=(0, 1, 2, 3, 7, 100))


def test_tiny_fp16_garbage_in_unused_slots():
    """Slots past each context hold NaN bit patterns; they must not leak in."""
    w = W.make("tiny_fp16")
    _run_full(w, splits_list=(0, 1, 3), fill=0xFF)


def test_llama8b_bf16_full():
    w = W.make("llama3_8b_bf16")
    _run_full(w, splits_list=(0, 1, 5))


def test_llama8b_fp8_steps():
    """FP8 cache with 1% x8 K outliers; 32 steps of (write one token per
    sequence, decode).  Cache bytes bit-exact, outputs within tolerance."""
    w = W.make("llama3_8b_fp8", steps=32)
    w.compute_fp8_scales()
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    fill_both(w, pool, op)
    tables = w.block_tables.copy()
    spare = list(w.spare_blocks)
    ctx = w.ctx_lens.copy()
    vmax = None
    for step in range(w.steps):
        # one new token per sequence at position ctx[s]
        ks, vs, slots = [], [], []
        for s in range(w.S):
            pos = int(ctx[s])
            if pos % 16 == 0:
                tables[s, pos // 16] = spare.pop(0)
            k, v = w.kv_bits(s, pos, pos + 1)
            ks.append(k)
            vs.append(v)
            slots.append(int(tables[s, pos // 16]) * 16 + pos % 16)
        k, v = np.concatenate(ks), np.concatenate(vs)
        slots = np.array(slots, np.int64)
        pool.reshape_and_cache(bits_to_torch(k, "bf16"), bits_to_torch(v, "bf16"),
                               torch.from_numpy(slots).cuda())
        oracle.reshape_and_cache("fp8_e4m3", w.num_blocks, 16, 8, 128, k, v, slots, w.k_scale,
                                 w.v_scale, *op)
        ctx = ctx + 1
        q = w.q_bits(step)
        out = gpu_decode(w, pool, q, ctx=ctx, tables=tables)
        if step in (0, 1, 15, 31):
            ref = oracle_decode(w, op, q, ctx=ctx, tables=tables)
            vmax = vmax_of(w, op)
            check_half(out, ref, vmax)
            if step == 31:
                check_fp32(gpu_decode(w, pool, q, ctx=ctx, tables=tables,
                                      out_dtype=torch.float32), ref)
    pool_bytes_equal(pool, op)
    assert pool.device_error() == N.PA_OK
    # the outliers saturate nothing under amax/448; codes reach +-448 only at amax
    kb = op[0]
    assert np.count_nonzero((kb & 0x7F) == 0x7E) >= 1


def test_llama8b_fp8_saturating_static_scale():
    """A static scale calibrated before the outliers were injected: ~1% of K
    codes saturate to +-448, still bit-exact."""
    w = W.make("llama3_8b_fp8", scale_down=4, steps=1)
    w.outlier_frac = 0.0
    w.compute_fp8_scales()
    w.outlier_frac = 0.01  # outliers now exceed the calibrated range
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    fill_both(w, pool, op)
    torch.cuda.synchronize()
    pool_bytes_equal(pool, op)
    sat = np.count_nonzero((op[0] & 0x7F) == 0x7E)
    assert sat > 0.002 * op[0].size * 0.25
    q = w.q_bits()
    ref = oracle_decode(w, op, q)
    check_half(gpu_decode(w, pool, q), ref, vmax_of(w, op))
    check_fp32(gpu_decode(w, pool, q, out_dtype=torch.float32), ref)


@pytest.mark.parametrize("name", ["llama3_70b_fp8_a", "llama3_70b_fp8_b"])
def test_llama70b_fp8_reduced(name):
    w = W.make(name, scale_down=16)
    _run_full(w, splits_list=(0, 1, 3))


def _compact(w, seqs):
    """Sampled sequences re-laid onto blocks 0..n-1 for the oracle (the output
    is invariant under relabelling physical blocks)."""
    ids = []
    for s in seqs:
        ids += list(w.block_tables[s, : -(-int(w.ctx_lens[s]) // 16)])
    remap = {b: i for i, b in enumerate(ids)}
    tables = np.zeros((len(seqs), w.max_blocks), np.int32)
    for r, s in enumerate(seqs):
        nb = -(-int(w.ctx_lens[s]) // 16)
        tables[r, :nb] = [remap[b] for b in w.block_tables[s, :nb]]
    return np.array(ids), tables


B_SAMPLE = sorted({0, 255} | set(int(x) for x in np.random.default_rng(1234).choice(256, 30,
                                                                                    replace=False)))


@pytest.mark.slow
@pytest.mark.parametrize("name,sample", [("llama3_70b_fp8_a", [0, 1, 2, 3]),
                                         ("llama3_70b_fp8_b", B_SAMPLE)])
def test_llama70b_fp8_full_size_sampled(name, sample):
    """Every sequence of the 4 x 131072 batch and 32 of the 256 x 4096 batch."""
    full_size_sampled_check(name, sample)


def test_permutation_invariance_bit_exact_on_gpu():
    """Relabelling physical blocks leaves the GPU output bit-identical."""
    w = W.make("llama3_70b_fp8_b", scale_down=8)
    w.compute_fp8_scales()
    pool = new_pool(w, 0)
    fill_both(w, pool, None)
    q = w.q_bits()
    out = gpu_decode(w, pool, q).cpu()
    perm = np.random.default_rng(21).permutation(w.num_blocks)
    pool2 = new_pool(w, 0)
    for which in ("k", "v"):
        src = pool.layer_view(which)
        dst = pool2.layer_view(which)
        dst[torch.from_numpy(perm).cuda()] = src
    tables2 = perm[w.block_tables].astype(np.int32)
    out2 = gpu_decode(w, pool2, q, tables=tables2).cpu()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_unit_values_give_unit_output():
    """V == 1 everywhere: every output is 1 up to fp32 rounding (softmax
    weights sum to one)."""
    w = W.make("llama3_8b_bf16", scale_down=4)
    pool = new_pool(w, 0)
    fill_both(w, pool, None)
    pool.v_cache.view(torch.int16).fill_(0x3F80)  # bf16 1.0
    out = gpu_decode(w, pool, w.q_bits(), out_dtype=torch.float32)
    assert torch.allclose(out, torch.ones_like(out), rtol=0, atol=2e-6)


def _hand_pool(kv_dtype, Hkv, d, nb, scale=1.0):
    p = KVPool(1, nb, Hkv, d, kv_dtype, scale, scale)
    p.k_cache.zero_()
    p.v_cache.zero_()
    return p


@pytest.mark.parametrize("kv_dtype", ["fp16", "bf16", "fp8_e4m3"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_shapes_and_ragged_contexts(kv_dtype, d, G):
    """Every dtype x head dim x group size, contexts around block boundaries
    (0, 1, 15, 16, 17, 31, 32, 33, a full table) and forced splits."""
    Hkv = 2
    ctx = np.array([0, 1, 15, 16, 17, 31, 32, 33, 200, 256], np.int32)
    max_blocks = 16
    nb = int(np.sum(-(-ctx // 16))) + 5
    rng = np.random.default_rng(G * 1000 + d)
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.zeros((len(ctx), max_blocks), np.int32)
    used = 0
    for s, n in enumerate(ctx):
        k = -(-int(n) // 16)
        tables[s, :k] = perm[used:used + k]
        tables[s, k:] = rng.integers(-5, 10**6, max_blocks - k)  # never read
        used += k
    w = W.Workload(name="shapes", index=7, kv_dtype=kv_dtype, n_q_heads=Hkv * G, n_kv_heads=Hkv,
                   head_dim=d, ctx_lens=ctx, num_blocks=nb, block_tables=tables)
    w.compute_fp8_scales()
    pool = new_pool(w, 0xFF)
    op = oracle_pools(w, 0xFF)
    fill_both(w, pool, op)
    q = w.q_bits()
    ref = oracle_decode(w, op, q)
    vmax = vmax_of(w, op)
    for ns in (0, 1, 4):
        out = gpu_decode(w, pool, q, num_splits=ns)
        check_half(out, ref, vmax)
        assert torch.all(out[0] == 0)  # empty context
        check_fp32(gpu_decode(w, pool, q, out_dtype=torch.float32, num_splits=ns), ref)
    assert pool.device_error() == N.PA_OK


def test_single_token_context_returns_v0_exactly():
    Hkv, d = 2, 128
    pool = _hand_pool("bf16", Hkv, d, 4)
    k = torch.randn(1, Hkv, d, dtype=torch.bfloat16, device="cuda")
    v = torch.randn(1, Hkv, d, dtype=torch.bfloat16, device="cuda")
    pool.reshape_and_cache(k, v, torch.tensor([3 * 16 + 0], dtype=torch.int64, device="cuda"))
    q = torch.randn(1, 8, d, dtype=torch.bfloat16, device="cuda")
    out = pool.decode(q, torch.tensor([[3]], dtype=torch.int32, device="cuda"),
                      torch.tensor([1], dtype=torch.int32, device="cuda"), out_dtype=torch.float32)
    ref = v.float().repeat_interleave(4, dim=1)
    assert torch.equal(out, ref)


def test_bounds_errors_are_reported_not_faulted():
    Hkv, d = 2, 64
    pool = _hand_pool("fp16", Hkv, d, 8)
    q = torch.randn(2, 4, d, dtype=torch.float16, device="cuda")
    tables = torch.tensor([[1, 2], [3, 9]], dtype=torch.int32, device="cuda")  # 9 >= 8
    ctx = torch.tensor([20, 20], dtype=torch.int32, device="cuda")
    pool.decode(q, tables, ctx)
    assert pool.device_error() == N.PA_ERR_BOUNDS
    ctx_long = torch.tensor([40, 3], dtype=torch.int32, device="cuda")  # > 2 blocks
    tables_ok = torch.tensor([[1, 2], [3, 4]], dtype=torch.int32, device="cuda")
    pool.decode(q, tables_ok, ctx_long)
    assert pool.device_error() == N.PA_ERR_BOUNDS
    pool.decode(q, tables_ok, torch.tensor([20, 3], dtype=torch.int32, device="cuda"))
    assert pool.device_error() == N.PA_OK


def test_host_validation():
    pool = _hand_pool("bf16", 2, 128, 8)
    q = torch.zeros(1, 6, 128, dtype=torch.bfloat16, device="cuda")   # 6 % 2 == 0, G = 3 ok
    t = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    c = torch.ones(1, dtype=torch.int32, device="cuda")
    pool.decode(q, t, c)
    with pytest.raises(N.PAError):
        pool.decode(torch.zeros(1, 5, 128, dtype=torch.bfloat16, device="cuda"), t, c)
    with pytest.raises(N.PAError):
        pool.decode(torch.zeros(1, 18, 128, dtype=torch.bfloat16, device="cuda"), t, c)  # G 9
    with pytest.raises(N.PAError):  # too little workspace for forced splits
        N.pa_decode(pool.handle, 0, q.data_ptr(), N.PA_BF16, q.data_ptr(), t.data_ptr(), 1,
                    c.data_ptr(), 1, 6, 1.0, 1, 0, 0, 0)
        N.pa_decode(pool.handle, 0, q.data_ptr(), N.PA_BF16, q.data_ptr(), t.data_ptr(), 64,
                    c.data_ptr(), 1, 6, 1.0, 8, 0, 0, 0)
    with pytest.raises(N.PAError):  # wrong output dtype
        N.pa_decode(pool.handle, 0, q.data_ptr(), N.PA_FP16, q.data_ptr(), t.data_ptr(), 1,
                    c.data_ptr(), 1, 6, 1.0, 1, 0, 0, 0)


def _prefix_share_setup(pool_blocks=4096):
    ps = W.PrefixShare()
    pool = KVPool(1, pool_blocks, 8, 128, "bf16")
    pool.k_cache.zero_()
    pool.v_cache.zero_()
    return ps, pool


def test_prefix_sharing_decode():
    """64 requests share a 2048-token prefix (128 refcounted blocks) plus their
    own U[128, 1024] suffix; tables come from the library's allocator and are
    checked against the reference model."""
    from oracle.allocator_model import AllocatorModel
    ps, pool = _prefix_share_setup()
    model = AllocatorModel(pool.num_blocks)
    prefix = pool.alloc(128)
    assert list(prefix) == model.alloc(128)
    suf = ps.suffix_lens()
    ctx = (2048 + suf).astype(np.int32)
    tables = np.zeros((ps.n_requests, -(-int(ctx.max()) // 16)), np.int32)
    op = (np.zeros(pool.k_cache.numel(), np.uint8), np.zeros(pool.v_cache.numel(), np.uint8))
    kp, vp = ps.prefix_kv()
    slots = prefix.astype(np.int64).repeat(16) * 16 + np.tile(np.arange(16), 128)
    pool.reshape_and_cache(bits_to_torch(kp, "bf16"), bits_to_torch(vp, "bf16"),
                           torch.from_numpy(slots).cuda())
    oracle.reshape_and_cache("bf16", pool.num_blocks, 16, 8, 128, kp, vp, slots, 1, 1, *op)
    for r in range(ps.n_requests):
        if r:
            pool.incref(prefix)
            model.incref(list(prefix))
        nb = -(-int(suf[r]) // 16)
        own = pool.alloc(nb)
        assert list(own) == model.alloc(nb)
        tables[r, :128] = prefix
        tables[r, 128:128 + nb] = own
        k, v = ps.suffix_kv(r, int(suf[r]))
        pos = np.arange(int(suf[r]))
        sl = own[pos // 16].astype(np.int64) * 16 + pos % 16
        pool.reshape_and_cache(bits_to_torch(k, "bf16"), bits_to_torch(v, "bf16"),
                               torch.from_numpy(sl).cuda())
        oracle.reshape_and_cache("bf16", pool.num_blocks, 16, 8, 128, k, v, sl, 1, 1, *op)
    assert pool.stats() == model.stats()
    assert pool.refcount(int(prefix[0])) == 64
    model.check_invariants([list(t[:-(-int(c) // 16)]) for t, c in zip(tables, ctx)])
    torch.cuda.synchronize()
    pool_bytes_equal(pool, op)
    q = ps.q_bits(ps.n_requests)
    w = W.Workload(name="prefix", index=4, kv_dtype="bf16", n_q_heads=32, n_kv_heads=8,
                   head_dim=128, ctx_lens=ctx, num_blocks=pool.num_blocks, block_tables=tables)
    ref = oracle_decode(w, op, q)
    check_half(gpu_decode(w, pool, q), ref, vmax_of(w, op))
    check_fp32(gpu_decode(w, pool, q, out_dtype=torch.float32), ref)


@pytest.mark.parametrize("prompt", [2000, 2008])
def test_best_of_8_branching_with_copy_on_write(prompt):
    """8 branches over one prompt; before its first append each branch whose
    tail block is shared gets a private copy (pa_cow_prepare + pa_copy_blocks);
    then 64 decode steps of (write one token per branch, decode)."""
    from oracle.allocator_model import AllocatorModel
    ps, pool = _prefix_share_setup(512)
    model = AllocatorModel(pool.num_blocks)
    nb = -(-prompt // 16)
    pblocks = pool.alloc(nb)
    assert list(pblocks) == model.alloc(nb)
    op = (np.zeros(pool.k_cache.numel(), np.uint8), np.zeros(pool.v_cache.numel(), np.uint8))
    kp, vp = ps.prefix_kv(prompt)
    pos = np.arange(prompt)
    slots = pblocks[pos // 16].astype(np.int64) * 16 + pos % 16
    pool.reshape_and_cache(bits_to_torch(kp, "bf16"), bits_to_torch(vp, "bf16"),
                           torch.from_numpy(slots).cuda())
    oracle.reshape_and_cache("bf16", pool.num_blocks, 16, 8, 128, kp, vp, slots, 1, 1, *op)
    width = -(-(prompt + 64) // 16)
    tables = np.zeros((8, width), np.int32)
    mtables = []
    for b in range(8):
        if b:
            pool.incref(pblocks)
            model.incref(list(pblocks))
        tables[b, :nb] = pblocks
        mtables.append(list(pblocks) + [0] * (width - nb))
    pairs = []
    for b in range(8):
        row = np.ascontiguousarray(tables[b])
        got = pool.cow_prepare(row, prompt)
        tables[b] = row
        want = model.cow_prepare(mtables[b], prompt)
        assert got == want
        if got:
            pairs.append(got)
    assert len(pairs) == (7 if prompt % 16 else 0)
    if pairs:
        pt = np.array(pairs, np.int32)
        pool.copy_blocks(torch.from_numpy(pt).cuda())
        oracle.copy_blocks("bf16", pool.num_blocks, 16, 8, 128, pt, *op)
    ctx = np.full(8, prompt, np.int32)
    w = W.Workload(name="branch", index=4, kv_dtype="bf16", n_q_heads=32, n_kv_heads=8,
                   head_dim=128, ctx_lens=ctx, num_blocks=pool.num_blocks, block_tables=tables)
    for step in range(64):
        new_slots = []
        for b in range(8):
            p = int(ctx[b])
            if p % 16 == 0:
                blk = pool.alloc(1)[0]
                assert blk == model.alloc(1)[0]
                tables[b, p // 16] = blk
                mtables[b][p // 16] = int(blk)
            new_slots.append(int(tables[b, p // 16]) * 16 + p % 16)
        k, v = ps.suffix_kv(1000 + step, 8)  # one new token for each branch
        sl = np.array(new_slots, np.int64)
        pool.reshape_and_cache(bits_to_torch(k, "bf16"), bits_to_torch(v, "bf16"),
                               torch.from_numpy(sl).cuda())
        oracle.reshape_and_cache("bf16", pool.num_blocks, 16, 8, 128, k, v, sl, 1, 1, *op)
        ctx = ctx + 1
        q = ps.q_bits(8, step)
        out = gpu_decode(w, pool, q, ctx=ctx, tables=tables)
        if step in (0, 63):
            ref = oracle_decode(w, op, q, ctx=ctx, tables=tables)
            check_half(out, ref, vmax_of(w, op))
    assert [list(t) for t in tables] == mtables
    assert pool.stats() == model.stats()
    expect_blocks = (126 + 7 + 32) if prompt % 16 else (125 + 32)
    assert pool.stats()[0] == expect_blocks
    torch.cuda.synchronize()
    pool_bytes_equal(pool, op)
    assert pool.device_error() == N.PA_OK
    for t in tables:
        pool.free(t[: -(-int(ctx[0]) // 16)])
    assert pool.stats() == (0, pool.num_blocks, 0)
