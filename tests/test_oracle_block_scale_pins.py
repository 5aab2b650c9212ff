"""Pins of the oracle's dynamic per-block FP8 scaling ("Optimización de KV Cache
con PagedAttention y Cuantización FP8 para Contextos Largos (128K)", section 8,
dynamic scaling: the MaxAbs of each block is taken at inference time).

Expected codes below are worked by hand from the OCP E4M3 definition (value =
(1 + m/8) * 2^(e-7)): 448 = 1.75 * 2^8 is code 0x7E, 224 = 1.75 * 2^7 is 0x76,
112 = 1.75 * 2^6 is 0x6E.  Scales are fl32(MaxAbs / 448), formed here with
numpy's IEEE float32 division."""
import numpy as np

from paged_kv_cache_270_gb300 import workloads as W

DT = "fp8_e4m3_block"


def _pools(oracle_mod, nb, H, d, fill=0):
    n = oracle_mod.pool_bytes(DT, nb, 16, H, d)
    return np.full(n, fill, np.uint8), np.full(n, fill, np.uint8)


def _tiles(oracle_mod, pool, nb, H, d):
    return pool[:oracle_mod.tiles_bytes(DT, nb, 16, H, d)].reshape(nb, H, 16, d)


def _const_tokens(vals, H, d):
    x = np.repeat(np.asarray(vals, np.float32)[:, None, None], H, 1).repeat(d, 2)
    return W.f32_to_bf16_bits(x)


def _write(oracle_mod, kp, vp, nb, H, d, k, v, slots):
    st = oracle_mod.reshape_and_cache(DT, nb, 16, H, d, k, v, np.asarray(slots, np.int64), 1.0,
                                      1.0, kp, vp)
    assert st == 0


def test_worked_example_growing_max_reencodes_earlier_rows(oracle_mod):
    """Tokens of all-1.0, all-2.0, all-4.0 appended one per call to block 1:
    each larger MaxAbs re-encodes the earlier rows (448 -> 224 -> 112)."""
    nb, H, d = 3, 2, 64
    kp, vp = _pools(oracle_mod, nb, H, d, fill=0xAB)
    expect_rows = [[0x7E], [0x76, 0x7E], [0x6E, 0x76, 0x7E]]
    for i, val in enumerate([1.0, 2.0, 4.0]):
        x = _const_tokens([val], H, d)
        _write(oracle_mod, kp, vp, nb, H, d, x, x, [16 + i])
        for pool in (kp, vp):
            t = _tiles(oracle_mod, pool, nb, H, d)
            for r, code in enumerate(expect_rows[i]):
                assert np.all(t[1, :, r, :] == code), (i, r)
            s = oracle_mod.tile_scales(DT, nb, 16, H, d, pool)
            assert np.all(s[1] == np.float32(val) / np.float32(448.0))
            assert np.all(t[0] == 0xAB) and np.all(t[2] == 0xAB)  # other blocks untouched


def test_worked_example_orders_and_one_call(oracle_mod):
    nb, H, d = 1, 1, 64
    # 2.0 first: the scale never grows, 1.0 lands on 224
    kp, vp = _pools(oracle_mod, nb, H, d)
    _write(oracle_mod, kp, vp, nb, H, d, _const_tokens([2.0], H, d), _const_tokens([2.0], H, d), [0])
    _write(oracle_mod, kp, vp, nb, H, d, _const_tokens([1.0], H, d), _const_tokens([1.0], H, d), [1])
    t = _tiles(oracle_mod, kp, nb, H, d)
    assert np.all(t[0, 0, 0] == 0x7E) and np.all(t[0, 0, 1] == 0x76)
    # 1.0 then 2.0 in ONE call (one run): the same codes as two calls with re-encoding
    kq, vq = _pools(oracle_mod, nb, H, d)
    x = _const_tokens([1.0, 2.0], H, d)
    _write(oracle_mod, kq, vq, nb, H, d, x, x, [0, 1])
    kr, vr = _pools(oracle_mod, nb, H, d)
    _write(oracle_mod, kr, vr, nb, H, d, x[:1], x[:1], [0])
    _write(oracle_mod, kr, vr, nb, H, d, x[1:], x[1:], [1])
    assert np.array_equal(kq, kr) and np.array_equal(vq, vr)
    assert np.all(_tiles(oracle_mod, kq, nb, H, d)[0, 0, 0] == 0x76)


def test_each_value_within_half_ulp_of_its_tiles_grid(oracle_mod):
    """Fresh tiles, random values: the tile's largest |x| is coded +-448 and
    every value decodes to within half an E4M3 step of x at the tile's scale
    (2^-4 |x| in the normal range, 2^-10 s below it)."""
    nb, H, d = 6, 2, 128
    rng = np.random.default_rng(0)
    n = 16 * nb
    gain = np.exp2(rng.uniform(-10, 6, size=(nb, 1, 1, 1))).astype(np.float32)
    x = (rng.standard_normal((nb, 16, H, d)).astype(np.float32) * gain).reshape(n, H, d)
    bits = W.f32_to_bf16_bits(x)
    xf = W.bits_to_f32(bits, "bf16").astype(np.float64).reshape(nb, 16, H, d).transpose(0, 2, 1, 3)
    kp, vp = _pools(oracle_mod, nb, H, d)
    _write(oracle_mod, kp, vp, nb, H, d, bits, bits, np.arange(n))
    table = oracle_mod.e4m3_table()
    for pool in (kp, vp):
        codes = _tiles(oracle_mod, pool, nb, H, d)
        s = oracle_mod.tile_scales(DT, nb, 16, H, d, pool).astype(np.float64)
        amax = np.abs(xf).max(axis=(2, 3))
        assert np.array_equal(s.astype(np.float32), amax.astype(np.float32) / np.float32(448.0))
        dec = table[codes] * s[:, :, None, None]
        bound = np.maximum(np.abs(xf) * 2.0**-4, s[:, :, None, None] * 2.0**-10) * (1 + 2.0**-20)
        assert np.all(np.abs(dec - xf) <= bound)
        at_max = np.abs(xf) == amax[:, :, None, None]
        assert np.all(np.isin(codes[at_max], [0x7E, 0xFE]))
        assert np.all((codes[at_max] == 0xFE) == (xf[at_max] < 0))


def test_dynamic_scaling_flushes_less_than_static(oracle_mod):
    """Blocks whose magnitudes differ by up to 2^16: one static per-tensor scale
    sends the small blocks into the E4M3 subnormals or to zero, the per-block
    scale keeps every block on its own grid (the page's precision claim)."""
    nb, H, d = 8, 2, 64
    rng = np.random.default_rng(1)
    n = 16 * nb
    gain = np.exp2(rng.uniform(-12, 4, size=(nb, 1, 1, 1))).astype(np.float32)
    x = (rng.standard_normal((nb, 16, H, d)).astype(np.float32) * gain).reshape(n, H, d)
    bits = W.f32_to_bf16_bits(x)
    xf = W.bits_to_f32(bits, "bf16").astype(np.float64).reshape(nb, 16, H, d).transpose(0, 2, 1, 3)
    table = oracle_mod.e4m3_table()
    # static
    st_scale = float(np.float32(np.abs(xf).max()) / np.float32(448.0))
    n_st = oracle_mod.pool_bytes("fp8_e4m3", nb, 16, H, d)
    ks, vs = np.zeros(n_st, np.uint8), np.zeros(n_st, np.uint8)
    oracle_mod.reshape_and_cache("fp8_e4m3", nb, 16, H, d, bits, bits, np.arange(n), st_scale,
                                 st_scale, ks, vs)
    dec_st = table[ks.reshape(nb, H, 16, d)] * st_scale
    # dynamic
    kp, vp = _pools(oracle_mod, nb, H, d)
    _write(oracle_mod, kp, vp, nb, H, d, bits, bits, np.arange(n))
    s = oracle_mod.tile_scales(DT, nb, 16, H, d, kp).astype(np.float64)
    dec_dy = table[_tiles(oracle_mod, kp, nb, H, d)] * s[:, :, None, None]
    rel_st = np.abs(dec_st - xf) / np.abs(xf)
    rel_dy = np.abs(dec_dy - xf) / np.abs(xf)
    flushed_st = np.sum((dec_st == 0) & (xf != 0))
    flushed_dy = np.sum((dec_dy == 0) & (xf != 0))
    assert flushed_dy * 10 < flushed_st
    assert rel_dy.mean() < 0.75 * rel_st.mean()


def test_run_at_offset_zero_starts_the_tile_afresh(oracle_mod):
    """A reused block: a run written at offset 0 ignores the old scale and codes."""
    nb, H, d = 2, 2, 64
    rng = np.random.default_rng(2)
    big = W.f32_to_bf16_bits(rng.standard_normal((16, H, d)).astype(np.float32) * 100)
    small = W.f32_to_bf16_bits(rng.standard_normal((4, H, d)).astype(np.float32))
    kp, vp = _pools(oracle_mod, nb, H, d)
    _write(oracle_mod, kp, vp, nb, H, d, big, big, np.arange(16, 32))
    old = _tiles(oracle_mod, kp, nb, H, d)[1].copy()
    _write(oracle_mod, kp, vp, nb, H, d, small, small, np.arange(16, 20))
    kf, vf = _pools(oracle_mod, nb, H, d)
    _write(oracle_mod, kf, vf, nb, H, d, small, small, np.arange(16, 20))
    t, tf = _tiles(oracle_mod, kp, nb, H, d), _tiles(oracle_mod, kf, nb, H, d)
    assert np.array_equal(t[1, :, :4], tf[1, :, :4])
    assert np.array_equal(t[1, :, 4:], old[:, 4:])          # stale rows are not touched
    assert np.array_equal(oracle_mod.tile_scales(DT, nb, 16, H, d, kp),
                          oracle_mod.tile_scales(DT, nb, 16, H, d, kf))


def test_zero_tile_then_values(oracle_mod):
    nb, H, d = 1, 1, 64
    kp, vp = _pools(oracle_mod, nb, H, d, fill=0x55)
    z = _const_tokens([0.0], H, d)
    _write(oracle_mod, kp, vp, nb, H, d, z, z, [0])
    assert oracle_mod.tile_scales(DT, nb, 16, H, d, kp)[0, 0] == 0.0
    assert np.all(_tiles(oracle_mod, kp, nb, H, d)[0, 0, 0] == 0)
    one = _const_tokens([1.0], H, d)
    _write(oracle_mod, kp, vp, nb, H, d, one, one, [1])
    t = _tiles(oracle_mod, kp, nb, H, d)
    assert np.all(t[0, 0, 0] == 0) and np.all(t[0, 0, 1] == 0x7E)
    assert oracle_mod.tile_scales(DT, nb, 16, H, d, kp)[0, 0] == np.float32(1) / np.float32(448)


def test_runs_split_at_skipped_slots_and_block_ends(oracle_mod):
    """One call with two runs (a skipped token between them, a block boundary
    inside the second) equals one call per run."""
    nb, H, d = 4, 2, 64
    rng = np.random.default_rng(3)
    x = W.f32_to_bf16_bits(rng.standard_normal((9, H, d)).astype(np.float32) * np.float32(3))
    slots = np.array([37, 38, 39, -1, 13, 14, 15, 48, 49], np.int64)
    ka, va = _pools(oracle_mod, nb, H, d)
    _write(oracle_mod, ka, va, nb, H, d, x, x, slots)
    kb, vb = _pools(oracle_mod, nb, H, d)
    for lo, hi in ((0, 3), (4, 7), (7, 9)):
        _write(oracle_mod, kb, vb, nb, H, d, x[lo:hi], x[lo:hi], slots[lo:hi])
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)


def test_attention_reads_each_tiles_own_scales(oracle_mod):
    """Decode over a block-scaled pool equals slab attention over the values
    decoded with each tile's K and V scale (blocks placed out of order)."""
    H, G, d = 2, 4, 64
    ctx = np.array([70, 33], np.int32)
    nb = 9
    tables = np.array([[7, 2, 5, 0, 8], [4, 1, 6, 3, 3]], np.int32)
    rng = np.random.default_rng(4)
    kp, vp = _pools(oracle_mod, nb, H, d)
    K, V = np.zeros((2, 80, H, d)), np.zeros((2, 80, H, d))
    for s, n in enumerate(ctx):
        gain = np.exp2(rng.uniform(-6, 6, size=(5, 1, 1, 1))).astype(np.float32)
        k = (rng.standard_normal((5, 16, H, d)).astype(np.float32) * gain).reshape(80, H, d)[:n]
        v = (rng.standard_normal((5, 16, H, d)).astype(np.float32) / gain).reshape(80, H, d)[:n]
        kb, vb = W.f32_to_bf16_bits(k), W.f32_to_bf16_bits(v)
        pos = np.arange(n)
        _write(oracle_mod, kp, vp, nb, H, d, kb, vb, tables[s, pos // 16] * 16 + pos % 16)
    table = oracle_mod.e4m3_table()
    tk, tv = _tiles(oracle_mod, kp, nb, H, d), _tiles(oracle_mod, vp, nb, H, d)
    sk = oracle_mod.tile_scales(DT, nb, 16, H, d, kp)
    sv = oracle_mod.tile_scales(DT, nb, 16, H, d, vp)
    for s, n in enumerate(ctx):
        for p in range(int(n)):
            b, o = tables[s, p // 16], p % 16
            K[s, p] = table[tk[b, :, o]] * sk[b][:, None]
            V[s, p] = table[tv[b, :, o]] * sv[b][:, None]
    q = W.f32_to_bf16_bits(rng.standard_normal((2, H * G, d)).astype(np.float32))
    out = oracle_mod.paged_attention(DT, "bf16", nb, 16, H, d, kp, vp, 1.0, 1.0, q, tables, ctx,
                                     0.125)
    ref = oracle_mod.slab_attention(K, V, W.bits_to_f32(q, "bf16").astype(np.float64), ctx, 0.125)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)
    # prefill with one-token chunks is the same decode
    pre = oracle_mod.paged_prefill(DT, "bf16", nb, 16, H, d, kp, vp, 1.0, 1.0, q,
                                   np.array([0, 1, 2], np.int32), tables, ctx, 0.125)
    assert np.array_equal(pre, out)


def test_copy_and_swap_carry_the_scales(oracle_mod):
    nb, H, d = 5, 2, 64
    rng = np.random.default_rng(5)
    x = W.f32_to_bf16_bits(rng.standard_normal((48, H, d)).astype(np.float32))
    kp, vp = _pools(oracle_mod, nb, H, d)
    _write(oracle_mod, kp, vp, nb, H, d, x, x[::-1].copy(), np.arange(48))
    assert oracle_mod.copy_blocks(DT, nb, 16, H, d, np.array([[1, 4]]), kp, vp) == 0
    for pool in (kp, vp):
        t = _tiles(oracle_mod, pool, nb, H, d)
        s = oracle_mod.tile_scales(DT, nb, 16, H, d, pool)
        assert np.array_equal(t[4], t[1]) and np.array_equal(s[4], s[1])
    buf = oracle_mod.swap_gather(DT, nb, 16, H, d, np.array([2, 0]), kp, vp)
    tile = H * 16 * d
    rec = 2 * tile + 16                  # 2 * H fp32 scales = 16 bytes, no padding
    assert buf.size == 2 * rec
    for i, b in enumerate((2, 0)):
        r = buf[i * rec:(i + 1) * rec]
        assert np.array_equal(r[:tile], kp[b * tile:(b + 1) * tile])
        assert np.array_equal(r[tile:2 * tile], vp[b * tile:(b + 1) * tile])
        sc = r[2 * tile:].view(np.float32)
        assert np.array_equal(sc[:H], oracle_mod.tile_scales(DT, nb, 16, H, d, kp)[b])
        assert np.array_equal(sc[H:], oracle_mod.tile_scales(DT, nb, 16, H, d, vp)[b])
    # one kv head: 8 bytes of scales, padded with zeros to 16
    kq, vq = _pools(oracle_mod, 2, 1, 64)
    y = W.f32_to_bf16_bits(rng.standard_normal((16, 1, 64)).astype(np.float32))
    _write(oracle_mod, kq, vq, 2, 1, 64, y, y, np.arange(16))
    b1 = oracle_mod.swap_gather(DT, 2, 16, 1, 64, np.array([0]), kq, vq)
    assert b1.size == 2 * 16 * 64 + 16 and np.all(b1[-8:] == 0)


def test_block_scaled_workload_names():
    w = W.make("llama3_70b_fp8_block_b", scale_down=64)
    base = W.make("llama3_70b_fp8_b", scale_down=64)
    assert w.kv_dtype == DT and w.elem_bytes == 1 and w.block_scaled
    assert np.array_equal(w.block_tables, base.block_tables)
    k0, v0 = w.kv_bits(0, 0, 40)
    k1, v1 = base.kv_bits(0, 0, 40)
    assert np.array_equal(k0, k1) and np.array_equal(v0, v1)
    pages = int(np.sum(-(-w.ctx_lens // 16)))
    assert w.kv_bytes() == base.kv_bytes() + pages * w.n_kv_heads * 8
