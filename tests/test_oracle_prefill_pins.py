"""Pins of the oracle's chunked-prefill routine: one-token chunks are decode
steps, a chunk split in two gives the same rows as one chunk, a query never
sees tokens after it, and an equal-logit case has a closed form."""
import numpy as np
import pytest

from paged_kv_cache_270_gb300 import workloads as W


def _filled(oracle_mod, w):
    nbytes = oracle_mod.pool_bytes(w.kv_dtype, w.num_blocks, 16, w.n_kv_heads, w.head_dim)
    kp, vp = np.zeros(nbytes, np.uint8), np.zeros(nbytes, np.uint8)
    for s in range(w.S):
        n = int(w.ctx_lens[s])
        k, v = w.kv_bits(s, 0, n)
        oracle_mod.reshape_and_cache(w.kv_dtype, w.num_blocks, 16, w.n_kv_heads, w.head_dim, k, v,
                                     w.slots(s, 0, n), 1.0, 1.0, kp, vp)
    return kp, vp


def _prefill(oracle_mod, w, kp, vp, q, q_start, ctx=None):
    return oracle_mod.paged_prefill(w.kv_dtype, w.in_dtype, w.num_blocks, 16, w.n_kv_heads,
                                    w.head_dim, kp, vp, 1.0, 1.0, q, q_start, w.block_tables,
                                    w.ctx_lens if ctx is None else ctx, w.softmax_scale)


def _queries(w, chunks, seed=3):
    rng = np.random.default_rng(seed)
    T = int(sum(chunks))
    q = rng.standard_normal((T, w.n_q_heads, w.head_dim)).astype(np.float16).view(np.uint16)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    return q, q_start


def test_one_token_chunks_equal_decode(oracle_mod):
    w = W.make("tiny_fp16")
    kp, vp = _filled(oracle_mod, w)
    q, q_start = _queries(w, [1] * w.S)
    pre = _prefill(oracle_mod, w, kp, vp, q, q_start)
    dec = oracle_mod.paged_attention("fp16", "fp16", w.num_blocks, 16, w.n_kv_heads, w.head_dim,
                                     kp, vp, 1.0, 1.0, q, w.block_tables, w.ctx_lens,
                                     w.softmax_scale)
    assert np.array_equal(pre, dec)


def test_every_row_is_a_decode_at_its_position(oracle_mod):
    """Row j of a chunk ending at ctx equals a decode with context ctx - C + j + 1."""
    w = W.make("tiny_fp16")
    kp, vp = _filled(oracle_mod, w)
    chunks = [5, 17, 1, 40]
    q, q_start = _queries(w, chunks)
    pre = _prefill(oracle_mod, w, kp, vp, q, q_start)
    for s, C in enumerate(chunks):
        for j in range(C):
            r = q_start[s] + j
            ctx = np.array([w.ctx_lens[s] - C + j + 1], np.int32)
            dec = oracle_mod.paged_attention("fp16", "fp16", w.num_blocks, 16, w.n_kv_heads,
                                             w.head_dim, kp, vp, 1.0, 1.0, q[r:r + 1],
                                             w.block_tables[s:s + 1], ctx, w.softmax_scale)
            assert np.array_equal(pre[r], dec[0])


def test_chunk_split_in_two_gives_same_rows(oracle_mod):
    w = W.make("tiny_fp16")
    kp, vp = _filled(oracle_mod, w)
    s, n = 3, int(w.ctx_lens[3])          # ctx 100
    q, q_start = _queries(w, [60])
    tables = w.block_tables[s:s + 1]
    one = oracle_mod.paged_prefill("fp16", "fp16", w.num_blocks, 16, 2, 64, kp, vp, 1, 1, q,
                                   np.array([0, 60], np.int32), tables, np.array([n], np.int32),
                                   w.softmax_scale)
    first = oracle_mod.paged_prefill("fp16", "fp16", w.num_blocks, 16, 2, 64, kp, vp, 1, 1,
                                     q[:25], np.array([0, 25], np.int32), tables,
                                     np.array([n - 35], np.int32), w.softmax_scale)
    second = oracle_mod.paged_prefill("fp16", "fp16", w.num_blocks, 16, 2, 64, kp, vp, 1, 1,
                                      q[25:], np.array([0, 35], np.int32), tables,
                                      np.array([n], np.int32), w.softmax_scale)
    assert np.array_equal(one, np.concatenate([first, second]))


def test_queries_do_not_see_later_tokens(oracle_mod):
    w = W.make("tiny_fp16")
    kp, vp = _filled(oracle_mod, w)
    chunks = [0, 0, 0, 30]                 # the last 30 of sequence 3's 100 tokens
    q, q_start = _queries(w, chunks)
    base = _prefill(oracle_mod, w, kp, vp, q, q_start)
    # corrupt the K and V of token 85 (a query at position >= 85 sees it)
    blk, off = w.block_tables[3, 85 // 16], 85 % 16
    K = kp.view(np.uint16).reshape(w.num_blocks, 2, 16, 64)
    V = vp.view(np.uint16).reshape(w.num_blocks, 2, 16, 64)
    K[blk, :, off, :] = np.float16(3.0).view(np.uint16)
    V[blk, :, off, :] = np.float16(-7.0).view(np.uint16)
    after = _prefill(oracle_mod, w, kp, vp, q, q_start)
    pos = 70 + np.arange(30)              # positions of the chunk's queries
    assert np.array_equal(after[pos < 85], base[pos < 85])
    assert np.all(np.any(after[pos >= 85] != base[pos >= 85], axis=(1, 2)))


def test_equal_keys_give_running_mean(oracle_mod):
    """All keys equal: query at position p averages V over tokens 0..p."""
    n, C = 40, 24
    w = W.Workload(name="hand", index=0, kv_dtype="fp16", n_q_heads=2, n_kv_heads=1, head_dim=64,
                   ctx_lens=np.array([n], np.int32), num_blocks=3,
                   block_tables=np.array([[2, 0, 1]], np.int32))
    nbytes = oracle_mod.pool_bytes("fp16", 3, 16, 1, 64)
    kp, vp = np.zeros(nbytes, np.uint8), np.zeros(nbytes, np.uint8)
    k = np.full((n, 1, 64), 0.5, np.float16).view(np.uint16)
    v = (np.arange(n, dtype=np.float16)[:, None, None] * np.ones((1, 1, 64), np.float16))
    oracle_mod.reshape_and_cache("fp16", 3, 16, 1, 64, k, v.view(np.uint16), w.slots(0, 0, n), 1,
                                 1, kp, vp)
    q, q_start = _queries(w, [C])
    out = _prefill(oracle_mod, w, kp, vp, q, q_start)
    for j in range(C):
        p = n - C + j
        assert np.allclose(out[j], p / 2.0, rtol=0, atol=1e-12)


def test_zero_scale_gives_mean_of_visible_values(oracle_mod):
    """softmax_scale 0: every visible key has logit 0, so query row p of a
    chunk is the mean of V over tokens 0 .. p of its kv head (and a decode row
    the mean over the whole context), computed here from the stored values."""
    w = W.make("tiny_fp16")
    kp, vp = _filled(oracle_mod, w)
    chunks = [3, 17, 1, 40]
    q, q_start = _queries(w, chunks)
    pre = oracle_mod.paged_prefill("fp16", "fp16", w.num_blocks, 16, w.n_kv_heads, w.head_dim,
                                   kp, vp, 1.0, 1.0, q, q_start, w.block_tables, w.ctx_lens, 0.0)
    dec = oracle_mod.paged_attention("fp16", "fp16", w.num_blocks, 16, w.n_kv_heads, w.head_dim,
                                     kp, vp, 1.0, 1.0, q[q_start[1:] - 1], w.block_tables,
                                     w.ctx_lens, 0.0)
    G = w.n_q_heads // w.n_kv_heads
    for s, C in enumerate(chunks):
        n = int(w.ctx_lens[s])
        _, v = w.kv_bits(s, 0, n)
        vals = v.view(np.float16).astype(np.float64)  # [n, Hkv, d]
        run = np.cumsum(vals, axis=0) / np.arange(1, n + 1)[:, None, None]
        for j in range(C):
            want = np.repeat(run[n - C + j], G, axis=0)  # query head g reads kv head g // G
            assert np.allclose(pre[q_start[s] + j], want, rtol=0, atol=1e-12)
        assert np.allclose(dec[s], np.repeat(run[n - 1], G, axis=0), rtol=0, atol=1e-12)


def test_negated_scale_equals_negated_queries(oracle_mod):
    """softmax(-s q.k) = softmax(s (-q).k): a negative score scale is the
    softmax of the negated scores, not of their magnitudes (negating fp16 q is
    exact, so the two calls agree bit for bit)."""
    w = W.make("tiny_fp16")
    kp, vp = _filled(oracle_mod, w)
    chunks = [4, 9, 1, 30]
    q, q_start = _queries(w, chunks)
    s = w.softmax_scale
    args = ("fp16", "fp16", w.num_blocks, 16, w.n_kv_heads, w.head_dim, kp, vp, 1.0, 1.0)
    a = oracle_mod.paged_prefill(*args, q, q_start, w.block_tables, w.ctx_lens, -s)
    b = oracle_mod.paged_prefill(*args, q ^ np.uint16(0x8000), q_start, w.block_tables,
                                 w.ctx_lens, s)
    c = oracle_mod.paged_prefill(*args, q, q_start, w.block_tables, w.ctx_lens, s)
    assert np.array_equal(a, b)
    assert not np.allclose(a, c)  # the sign matters


def test_invalid_chunk_rejected(oracle_mod):
    w = W.make("tiny_fp16")
    kp, vp = _filled(oracle_mod, w)
    q, q_start = _queries(w, [1, 1, 1, 101])   # chunk longer than the context
    with pytest.raises(ValueError):
        _prefill(oracle_mod, w, kp, vp, q, q_start)


def _tiny_of_kind(kv_dtype):
    w = W.make("tiny_fp16")
    w.kv_dtype = kv_dtype
    if kv_dtype == "fp8_e4m3":
        w.k_scale, w.v_scale = 2.0 ** -5, 2.0 ** -5  # N(0,1) values span many E4M3 binades
    return w


def _filled_kind(oracle_mod, w):
    nbytes = oracle_mod.pool_bytes(w.kv_dtype, w.num_blocks, 16, w.n_kv_heads, w.head_dim)
    kp, vp = np.zeros(nbytes, np.uint8), np.zeros(nbytes, np.uint8)
    for s in range(w.S):
        n = int(w.ctx_lens[s])
        for lo in range(0, n, 7):  # several calls per sequence: block-scaled tiles re-encode
            k, v = w.kv_bits(s, lo, min(n, lo + 7))
            assert oracle_mod.reshape_and_cache(w.kv_dtype, w.num_blocks, 16, w.n_kv_heads,
                                                w.head_dim, k, v, w.slots(s, lo, min(n, lo + 7)),
                                                w.k_scale, w.v_scale, kp, vp) == 0
    return kp, vp


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "fp8_e4m3_block"])
def test_rows_are_decodes_for_every_pool_kind(oracle_mod, kv_dtype):
    """On every pool kind, row j of a chunk ending at ctx equals a decode with
    context ctx - C + j + 1 (one-token chunks are plain decode steps)."""
    w = _tiny_of_kind(kv_dtype)
    kp, vp = _filled_kind(oracle_mod, w)
    chunks = [1, 17, 5, 40]
    rng = np.random.default_rng(11)
    q = W.f32_to_bf16_bits(rng.standard_normal((sum(chunks), w.n_q_heads, w.head_dim),
                                               dtype=np.float32))
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    args = (kv_dtype, "bf16", w.num_blocks, 16, w.n_kv_heads, w.head_dim, kp, vp, w.k_scale,
            w.v_scale)
    pre = oracle_mod.paged_prefill(*args, q, q_start, w.block_tables, w.ctx_lens,
                                   w.softmax_scale)
    for s, C in enumerate(chunks):
        for j in range(C):
            r = q_start[s] + j
            ctx = np.array([w.ctx_lens[s] - C + j + 1], np.int32)
            dec = oracle_mod.paged_attention(*args, q[r:r + 1], w.block_tables[s:s + 1], ctx,
                                             w.softmax_scale)
            assert np.array_equal(pre[r], dec[0])
