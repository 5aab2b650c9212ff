"""GPU parity of block-scaled FP8 pools (a dynamic scale per (block, kv head)
tile, "Optimización de KV Cache con PagedAttention y Cuantización FP8 para
Contextos Largos (128K)", section 8, dynamic scaling) against the fp64 oracle:
the written codes and scales bit for bit, decode and prefill within the stated
tolerances, block copies and swaps carrying the scales."""
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
DT = "fp8_e4m3_block"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_270_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    oracle.build()


def _workload(d, G, ctx, seed, Hkv=2, extra_blocks=3):
    ctx = np.asarray(ctx, np.int32)
    max_blocks = int(max(1, -(-int(ctx.max()) // 16)))
    nb = int(np.sum(-(-ctx // 16))) + extra_blocks
    rng = np.random.default_rng(seed)
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.zeros((len(ctx), max_blocks), np.int32)
    used = 0
    for s, n in enumerate(ctx):
        k = -(-int(n) // 16)
        tables[s, :k] = perm[used:used + k]
        used += k
    return W.Workload(name=f"block_{d}_{G}", index=11, kv_dtype=DT, n_q_heads=Hkv * G,
                      n_kv_heads=Hkv, head_dim=d, ctx_lens=ctx, num_blocks=nb,
                      block_tables=tables, kv_seed=seed)


def _gained(w, s, lo, hi, rng):
    """K/V of tokens [lo, hi) of sequence s, each token scaled by its own gain
    (log-uniform over 2^-4 .. 2^4), so later tokens often raise a tile's MaxAbs."""
    k, v = w.kv_bits(s, lo, hi)
    g = np.exp2(rng.uniform(-4, 4, size=(hi - lo, 1, 1))).astype(np.float32)
    kf = W.bits_to_f32(k, "bf16") * g
    vf = W.bits_to_f32(v, "bf16") / g
    return W.f32_to_bf16_bits(kf), W.f32_to_bf16_bits(vf)


def _write_both(w, pool, op, k, v, slots):
    pool.reshape_and_cache(bits_to_torch(k, "bf16"), bits_to_torch(v, "bf16"),
                           torch.from_numpy(np.asarray(slots, np.int64)).cuda())
    st = oracle.reshape_and_cache(DT, w.num_blocks, 16, w.n_kv_heads, w.head_dim, k, v,
                                  np.asarray(slots, np.int64), 1.0, 1.0, *op)
    return st


def _fill_in_pieces(w, pool, op, seed, max_piece=40, pad=True):
    """Write every sequence's tokens in random pieces (1 .. max_piece tokens),
    several sequences per call in random order, with skipped (-1) padding
    tokens between them: runs start inside blocks and grow their MaxAbs."""
    rng = np.random.default_rng(seed)
    done = np.zeros(w.S, np.int64)
    written = [([], []) for _ in range(w.S)]  # each sequence's values, in write order
    while np.any(done < w.ctx_lens):
        live = np.flatnonzero(done < w.ctx_lens)
        pick = rng.permutation(live)[:rng.integers(1, len(live) + 1)]
        ks, vs, slots = [], [], []
        for s in pick:
            lo = int(done[s])
            hi = min(int(w.ctx_lens[s]), lo + int(rng.integers(1, max_piece + 1)))
            k, v = _gained(w, s, lo, hi, rng)
            written[s][0].append(k)
            written[s][1].append(v)
            pos = np.arange(lo, hi)
            ks.append(k)
            vs.append(v)
            slots.append(w.block_tables[s, pos // 16].astype(np.int64) * 16 + pos % 16)
            if pad and rng.random() < 0.3:
                z = np.zeros((1, w.n_kv_heads, w.head_dim), np.uint16)
                ks.append(z)
                vs.append(z)
                slots.append(np.array([-1], np.int64))
            done[s] = hi
        assert _write_both(w, pool, op, np.concatenate(ks), np.concatenate(vs),
                           np.concatenate(slots)) == 0
    return [(np.concatenate(a), np.concatenate(b)) for a, b in written]


@pytest.mark.parametrize("d,Hkv", [(64, 1), (64, 8), (128, 2), (128, 8)])
def test_writes_in_pieces_bit_exact(d, Hkv):
    w = _workload(d, 1, [1, 15, 16, 17, 40, 100, 333], seed=d + Hkv, Hkv=Hkv)
    pool = new_pool(w, 0xFF)
    op = oracle_pools(w, 0xFF)
    values = _fill_in_pieces(w, pool, op, seed=d * Hkv)
    torch.cuda.synchronize()
    used = np.concatenate([w.block_tables[s, :-(-int(n) // 16)] for s, n in enumerate(w.ctx_lens)])
    pool_bytes_equal(pool, op, blocks=used)
    assert pool.device_error() == N.PA_OK
    # The same values written one sequence per call: every tile ends with the
    # same scale fl32(MaxAbs / 448), while the piecewise pool's codes differ
    # where a growing MaxAbs re-encoded earlier rows -- so that path ran.
    one = oracle_pools(w, 0xFF)
    for s_, (k, v) in enumerate(values):
        assert oracle.reshape_and_cache(DT, w.num_blocks, 16, Hkv, d, k, v,
                                        w.slots(s_, 0, int(w.ctx_lens[s_])), 1.0, 1.0, *one) == 0
    for a, b in zip(op, one):
        sa = oracle.tile_scales(DT, w.num_blocks, 16, Hkv, d, a)[used]
        sb = oracle.tile_scales(DT, w.num_blocks, 16, Hkv, d, b)[used]
        assert np.array_equal(sa, sb)
    assert not np.array_equal(op[0], one[0])


def test_block_reuse_zero_tiles_and_bounds():
    w = _workload(128, 1, [64], seed=3, Hkv=2)
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    rng = np.random.default_rng(7)
    k, v = _gained(w, 0, 0, 64, rng)
    slots = w.slots(0, 0, 64)
    _write_both(w, pool, op, k, v, slots)
    # the sequence ends; its blocks are reused by a new one: runs at offset 0 start afresh
    k2, v2 = W.f32_to_bf16_bits(rng.standard_normal((20, 2, 128)).astype(np.float32) * 1e-3), \
        W.f32_to_bf16_bits(rng.standard_normal((20, 2, 128)).astype(np.float32) * 1e3)
    _write_both(w, pool, op, k2, v2, slots[:20])
    # an all-zero token opens a tile (scale 0), then real values append to it
    z = np.zeros((1, 2, 128), np.uint16)
    last = int(w.block_tables[0, 3]) * 16
    _write_both(w, pool, op, z, z, [last])
    _write_both(w, pool, op, k[:3], v[:3], [last + 1, last + 2, last + 3])
    torch.cuda.synchronize()
    pool_bytes_equal(pool, op, blocks=w.block_tables[0, :4])
    assert pool.device_error() == N.PA_OK
    # a slot past the pool is skipped and reported; the valid token is written
    bad = np.array([w.num_blocks * 16 + 5, int(w.block_tables[0, 2]) * 16], np.int64)
    pool.reshape_and_cache(bits_to_torch(k[:2], "bf16"), bits_to_torch(v[:2], "bf16"),
                           torch.from_numpy(bad).cuda())
    assert pool.device_error() == N.PA_ERR_BOUNDS
    oracle.reshape_and_cache(DT, w.num_blocks, 16, 2, 128, k[1:2], v[1:2], bad[1:], 1.0, 1.0, *op)
    pool_bytes_equal(pool, op, blocks=w.block_tables[0, :4])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_decode_parity(d, G):
    w = _workload(d, G, [1, 16, 17, 100, 257, 700], seed=G * 10 + d, Hkv=2)
    pool = new_pool(w, 0xFF)
    op = oracle_pools(w, 0xFF)
    _fill_in_pieces(w, pool, op, seed=G + d)
    q = w.q_bits()
    ref = oracle_decode(w, op, q)
    vmax = vmax_of(w, op)
    for ns in (0, 1, 3):
        check_half(gpu_decode(w, pool, q, num_splits=ns), ref, vmax)
        check_fp32(gpu_decode(w, pool, q, out_dtype=torch.float32, num_splits=ns), ref)
    assert pool.device_error() == N.PA_OK


def test_decode_steps_8b_shapes():
    """Llama-3-8B shapes: 24 steps of (append one token per sequence, decode);
    every append may re-encode its tile; codes, scales and outputs checked."""
    w = W.make("llama3_8b_fp8_block", scale_down=8, steps=24)
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    fill_both(w, pool, op)
    tables = w.block_tables.copy()
    spare = list(w.spare_blocks)
    ctx = w.ctx_lens.copy()
    rng = np.random.default_rng(9)
    for step in range(w.steps):
        ks, vs, slots = [], [], []
        for s in range(w.S):
            pos = int(ctx[s])
            if pos % 16 == 0:
                tables[s, pos // 16] = spare.pop(0)
            k, v = _gained(w, s, pos, pos + 1, rng)
            ks.append(k)
            vs.append(v)
            slots.append(int(tables[s, pos // 16]) * 16 + pos % 16)
        _write_both(w, pool, op, np.concatenate(ks), np.concatenate(vs), slots)
        ctx = ctx + 1
        q = w.q_bits(step)
        if step in (0, 7, 23):
            ref = oracle_decode(w, op, q, ctx=ctx, tables=tables)
            check_half(gpu_decode(w, pool, q, ctx=ctx, tables=tables), ref, vmax_of(w, op))
            check_fp32(gpu_decode(w, pool, q, ctx=ctx, tables=tables, out_dtype=torch.float32), ref)
    torch.cuda.synchronize()
    pool_bytes_equal(pool, op)
    assert pool.device_error() == N.PA_OK


@pytest.mark.parametrize("name", ["llama3_70b_fp8_block_a", "llama3_70b_fp8_block_b"])
def test_llama70b_block_reduced(name):
    """Both register builds of the block-scaled kernel: launches of at most four
    CTAs per SM (152 SMs) take the spill-free one, 32 forced splits (1024 and
    2048 CTAs here) the five-per-SM one."""
    w = W.make(name, scale_down=16)
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    fill_both(w, pool, op)
    q = w.q_bits()
    ref = oracle_decode(w, op, q)
    vmax = vmax_of(w, op)
    assert w.S * w.n_kv_heads * min(32, w.max_blocks) > 4 * 152
    for ns in (0, 1, 3, 32):
        check_half(gpu_decode(w, pool, q, num_splits=ns), ref, vmax)
        check_fp32(gpu_decode(w, pool, q, out_dtype=torch.float32, num_splits=ns), ref)
    torch.cuda.synchronize()
    pool_bytes_equal(pool, op)
    assert pool.device_error() == N.PA_OK


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_prefill_parity(d, G):
    pairs = [(0, 1), (0, 17), (5, 16), (30, 33), (100, 100), (200, 3)]
    ctx = [h + c for h, c in pairs]
    chunks = [c for _, c in pairs]
    w = _workload(d, G, ctx, seed=G * 7 + d, Hkv=2)
    pool = new_pool(w, 0xFF)
    op = oracle_pools(w, 0xFF)
    _fill_in_pieces(w, pool, op, seed=G * 3 + d)
    rng = np.random.default_rng(G + d)
    T = sum(chunks)
    q = W.f32_to_bf16_bits(rng.standard_normal((T, w.n_q_heads, d)).astype(np.float32))
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    ref = oracle.paged_prefill(DT, "bf16", w.num_blocks, 16, w.n_kv_heads, d, op[0], op[1], 1.0,
                               1.0, q, q_start, w.block_tables, w.ctx_lens, w.softmax_scale)
    args = (bits_to_torch(q, "bf16"), torch.from_numpy(q_start).cuda(),
            torch.from_numpy(w.block_tables).cuda(), torch.from_numpy(w.ctx_lens).cuda())
    out = pool.prefill(*args, max_chunk=max(chunks), softmax_scale=w.softmax_scale)
    out32 = pool.prefill(*args, max_chunk=max(chunks), softmax_scale=w.softmax_scale,
                         out_dtype=torch.float32)
    torch.cuda.synchronize()
    check_half(out, ref, vmax_of(w, op))
    check_fp32(out32, ref)
    assert pool.device_error() == N.PA_OK


def test_copy_and_swap_carry_scales():
    w = _workload(128, 4, [40, 90], seed=21, Hkv=8, extra_blocks=6)
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    _fill_in_pieces(w, pool, op, seed=22)
    src = w.block_tables[1, :3]
    dst = np.array([w.num_blocks - 1, w.num_blocks - 2, w.num_blocks - 3], np.int32)
    pairs = np.stack([src, dst], 1).astype(np.int32)
    pool.copy_blocks(torch.from_numpy(pairs.copy()).cuda())
    oracle.copy_blocks(DT, w.num_blocks, 16, 8, 128, pairs, *op)
    torch.cuda.synchronize()
    pool_bytes_equal(pool, op)
    # swap out: the host records equal the oracle's gather (tiles, scales, padding)
    rec = pool.swap_block_bytes()
    assert rec == 2 * 8 * 16 * 128 + 64
    ids = np.concatenate([w.block_tables[0, :3], dst]).astype(np.int32)
    host = torch.empty(rec * len(ids), dtype=torch.uint8).pin_memory()
    host.fill_(0x5A)
    pool.swap_out(torch.from_numpy(ids).cuda(), host)
    torch.cuda.synchronize()
    ref = oracle.swap_gather(DT, w.num_blocks, 16, 8, 128, ids, *op)
    assert np.array_equal(host.numpy(), ref)
    # swap back into other blocks: tiles and scales restored bit for bit
    other = KVPool(1, w.num_blocks, 8, 128, DT)
    other.k_cache.fill_(0xFF)
    other.v_cache.fill_(0xFF)
    other.swap_in(torch.from_numpy(ids).cuda(), host)
    torch.cuda.synchronize()
    for which in ("k", "v"):
        assert torch.equal(other.layer_view(which)[ids.tolist()], pool.layer_view(which)[ids.tolist()])
        assert torch.equal(other.scale_view(which)[ids.tolist()], pool.scale_view(which)[ids.tolist()])
    assert pool.device_error() == N.PA_OK


def test_multi_layer_scales_stay_in_their_layer():
    """A 3-layer pool: each layer's writes land in that layer's tiles and scale
    table only; decode of each layer matches the oracle."""
    L, nb, H, d = 3, 12, 2, 64
    pool = KVPool(L, nb, H, d, DT)
    pool.k_cache.fill_(0)
    pool.v_cache.fill_(0)
    rng = np.random.default_rng(5)
    refs = []
    for layer in range(L):
        k = W.f32_to_bf16_bits(rng.standard_normal((40, H, d)).astype(np.float32) * (layer + 1))
        v = W.f32_to_bf16_bits(rng.standard_normal((40, H, d)).astype(np.float32) / (layer + 1))
        slots = np.arange(16 * layer, 16 * layer + 40, dtype=np.int64)
        pool.reshape_and_cache(bits_to_torch(k, "bf16"), bits_to_torch(v, "bf16"),
                               torch.from_numpy(slots).cuda(), layer=layer)
        op = (np.zeros(oracle.pool_bytes(DT, nb, 16, H, d), np.uint8),
              np.zeros(oracle.pool_bytes(DT, nb, 16, H, d), np.uint8))
        oracle.reshape_and_cache(DT, nb, 16, H, d, k, v, slots, 1.0, 1.0, *op)
        refs.append(op)
    torch.cuda.synchronize()
    for layer, op in enumerate(refs):
        for which, o in (("k", op[0]), ("v", op[1])):
            assert np.array_equal(pool.layer_view(which, layer).cpu().numpy().ravel(),
                                  o[:nb * H * 16 * d])
            assert np.array_equal(pool.scale_view(which, layer).cpu().numpy(),
                                  oracle.tile_scales(DT, nb, 16, H, d, o))
        tables = np.arange(layer, layer + 3, dtype=np.int32)[None]
        q = W.f32_to_bf16_bits(rng.standard_normal((1, H * 4, d)).astype(np.float32))
        ctx = np.array([40], np.int32)
        ref = oracle.paged_attention(DT, "bf16", nb, 16, H, d, op[0], op[1], 1.0, 1.0, q, tables,
                                     ctx, 0.125)
        out = pool.decode(bits_to_torch(q, "bf16"), torch.from_numpy(tables).cuda(),
                          torch.from_numpy(ctx).cuda(), out_dtype=torch.float32,
                          softmax_scale=0.125, layer=layer)
        check_fp32(out, ref)
    assert pool.device_error() == N.PA_OK


@pytest.mark.slow
@pytest.mark.parametrize("name,sample", [("llama3_70b_fp8_block_a", [0, 1, 2, 3]),
                                         ("llama3_70b_fp8_block_b", [0, 77, 128, 255])])
def test_llama70b_block_full_size_sampled(name, sample):
    """Block-scaled FP8 at the benchmark's full sizes: every sequence of the 4 x
    131072 batch (19 automatic splits: the one-wave launch that takes the
    four-CTA register build) and sampled sequences of the 256 x 4096 batch,
    tiles and scales bit for bit, outputs within tolerance, both schedules."""
    full_size_sampled_check(name, sample)


def test_no_alloc_entry_point_on_block_scaled_pools():
    """pa_decode_no_alloc on a block-scaled pool gives exactly pa_decode's
    result for the same split count (same kernels, partials in the fixed array)."""
    w = W.make("llama3_70b_fp8_block_a", scale_down=32)
    pool = new_pool(w, 0)
    fill_both(w, pool, None)
    q = bits_to_torch(w.q_bits(), "bf16")
    t = torch.from_numpy(np.ascontiguousarray(w.block_tables)).cuda()
    c = torch.from_numpy(np.ascontiguousarray(w.ctx_lens)).cuda()
    S, Hq, D = q.shape
    stream = torch.cuda.current_stream().cuda_stream
    for ns in (1, 6):
        ws_bytes = N.pa_decode_workspace_bytes(pool.handle, S, Hq, t.shape[1], ns)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
        ref = torch.empty((S, Hq, D), dtype=torch.float32, device="cuda")
        got = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        N.pa_decode(pool.handle, 0, ref.data_ptr(), N.PA_FP32, q.data_ptr(), t.data_ptr(),
                    t.shape[1], c.data_ptr(), S, Hq, w.softmax_scale, ns, ws.data_ptr(), ws_bytes,
                    stream)
        N.pa_decode_no_alloc(pool.handle, 0, got.data_ptr(), N.PA_FP32, q.data_ptr(),
                             t.data_ptr(), t.shape[1], c.data_ptr(), S, Hq, w.softmax_scale, ns,
                             stream)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
    assert pool.device_error() == N.PA_OK


@pytest.mark.parametrize("H", [1, 2])
def test_swap_records_across_layers_carry_each_layers_scales(H):
    """3 layers: a swap record is the tiles of every layer then the scales
    [layer][K|V][head] and zero padding to 16 bytes (8 bytes of it with one kv
    head); swapping back into other blocks restores tiles and scales of every layer."""
    L, nb, d = 3, 10, 64
    pool = KVPool(L, nb, H, d, DT)
    pool.k_cache.fill_(0)
    pool.v_cache.fill_(0)
    rng = np.random.default_rng(11)
    for layer in range(L):
        k = W.f32_to_bf16_bits(rng.standard_normal((48, H, d)).astype(np.float32) * (layer + 1))
        v = W.f32_to_bf16_bits(rng.standard_normal((48, H, d)).astype(np.float32) * (layer + 3))
        pool.reshape_and_cache(bits_to_torch(k, "bf16"), bits_to_torch(v, "bf16"),
                               torch.arange(48, dtype=torch.int64, device="cuda"), layer=layer)
    ids = torch.tensor([2, 0], dtype=torch.int32, device="cuda")
    rec = pool.swap_block_bytes()
    tile = H * 16 * d
    scale_bytes = 2 * L * H * 4
    assert rec == 2 * L * tile + -(-scale_bytes // 16) * 16
    host = torch.empty(rec * 2, dtype=torch.uint8).pin_memory()
    host.fill_(0x77)
    pool.swap_out(ids, host)
    torch.cuda.synchronize()
    hb = host.numpy()
    for i, b in enumerate((2, 0)):
        r = hb[i * rec:(i + 1) * rec]
        sc = r[2 * L * tile:2 * L * tile + scale_bytes].view(np.float32).reshape(L, 2, H)
        for layer in range(L):
            base = 2 * layer * tile
            assert np.array_equal(r[base:base + tile],
                                  pool.layer_view("k", layer)[b].cpu().numpy().ravel())
            assert np.array_equal(r[base + tile:base + 2 * tile],
                                  pool.layer_view("v", layer)[b].cpu().numpy().ravel())
            assert np.array_equal(sc[layer, 0], pool.scale_view("k", layer)[b].cpu().numpy())
            assert np.array_equal(sc[layer, 1], pool.scale_view("v", layer)[b].cpu().numpy())
        assert np.all(r[2 * L * tile + scale_bytes:] == 0)   # padding is written as zeros
    dst = torch.tensor([7, 9], dtype=torch.int32, device="cuda")
    pool.swap_in(dst, host)
    torch.cuda.synchronize()
    for layer in range(L):
        for which in ("k", "v"):
            assert torch.equal(pool.layer_view(which, layer)[[7, 9]], pool.layer_view(which, layer)[[2, 0]])
            assert torch.equal(pool.scale_view(which, layer)[[7, 9]], pool.scale_view(which, layer)[[2, 0]])
    assert pool.device_error() == N.PA_OK
