"""Pins of the fp64 oracle against facts fixed outside it.

Each test ties one oracle routine to something it does not compute itself:
values the pages print (tests/golden/), closed forms, invariances of the
method, special cases with known answers, library routines (numpy's binary16,
torch's bfloat16 and float8_e4m3fn casts) and brute force.  A plausible bug in
the oracle -- a dropped term, a wrong index or sign, a transposed operand, a
wrong rounding tie -- fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from conftest import golden_lines
from paged_kv_cache_270_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ------------------------------------------------------------ (1) closed form
def test_bytes_per_token_matches_pages(oracle_mod):
    rows = golden_lines("kv_bytes_per_token.txt")
    assert rows
    for L, H, d, b, expect in rows:
        assert oracle_mod.kv_bytes_per_token(int(L), int(H), int(d), int(b)) == int(expect)


def test_session_sizes_exact_and_page_rounding(oracle_mod):
    per_tok = oracle_mod.kv_bytes_per_token(80, 8, 128, 2)
    for tokens, exact, printed_gb in golden_lines("session_sizes.txt"):
        assert int(tokens) * per_tok == int(exact)
        # the page's figures come from a rounded 0.32 MB/token
        assert abs(int(tokens) * 0.32e6 / 1e9 - float(printed_gb)) < 0.011


def test_pool_bytes_equal_closed_form_for_every_workload(oracle_mod):
    for name in ("tiny_fp16", "llama3_8b_bf16", "llama3_8b_fp8", "llama3_70b_fp8_a",
                 "llama3_70b_fp8_b"):
        w = W.make(name, scale_down=16)
        b = oracle_mod.pool_bytes(w.kv_dtype, w.num_blocks, 16, w.n_kv_heads, w.head_dim)
        per_tok = oracle_mod.kv_bytes_per_token(1, w.n_kv_heads, w.head_dim, w.elem_bytes)
        assert 2 * b == per_tok * w.num_blocks * 16


# ------------------------------------------------------------ number formats
def test_f16_decode_matches_numpy_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle_mod.value16("fp16", bits)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_decode_matches_torch_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle_mod.value16("bf16", bits)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_e4m3_special_values(oracle_mod):
    for code, val in golden_lines("e4m3_values.txt"):
        got = oracle_mod.e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val)
            assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e4m3_decode_matches_torch_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle_mod.e4m3_table()
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.isnan(got).sum() == 2  # only S.1111.111


def _bruteforce_e4m3(y: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code by exhaustive search over the finite grid; ties go to
    the even mantissa; magnitudes above 448 saturate to 448; sign kept."""
    mags = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()  # codes 0x00..0x7E
    codes = np.arange(0x7F)
    a = np.abs(y.astype(np.float64))
    dist = np.abs(a[:, None] - mags[None, :])
    tie = dist == dist.min(axis=1, keepdims=True)
    even_tie = tie & (codes[None, :] % 2 == 0)
    pick = np.where(even_tie.any(axis=1), even_tie.argmax(axis=1), tie.argmax(axis=1))
    assert np.all(tie.sum(axis=1)[a <= 448] <= 2)
    pick = np.where(a > 448, 0x7E, pick)
    return (pick | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


def _bf16_all_finite():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    keep = np.isfinite(f)
    return bits[keep], f[keep]


@pytest.mark.parametrize("scale", [1.0, 0.125, float(np.float32(4.75) / np.float32(448.0))])
def test_e4m3_quantiser_bruteforce_all_bf16(oracle_mod, scale):
    """code(x) == nearest grid point of fl32(x / s), for every finite bf16 x."""
    bits, x = _bf16_all_finite()
    y = (x.astype(np.float32) / np.float32(scale)).astype(np.float32)  # IEEE fp32 division
    want = _bruteforce_e4m3(y)
    got = np.array([oracle_mod.quantize_e4m3(float(v), scale) for v in x], np.uint8)
    assert np.array_equal(got, want)


def test_e4m3_quantiser_matches_torch_cast_in_range(oracle_mod):
    """Within +-448 torch's float8_e4m3fn cast is RNE; compare all bf16 values."""
    bits, x = _bf16_all_finite()
    keep = np.abs(x) <= 448
    x = x[keep]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.e4m3_encode(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_ties_saturation_and_sign(oracle_mod):
    enc = oracle_mod.e4m3_encode
    # midpoints between grid neighbours go to the even mantissa
    assert enc(1.0625) == 0x38      # between 1.0 (m=0) and 1.125 (m=1): even -> 1.0
    assert enc(1.1875) == 0x3A      # between 1.125 (m=1) and 1.25 (m=2): even -> 1.25
    assert enc(2.0 ** -10) == 0x00  # half of the smallest subnormal: even -> 0
    assert enc(3 * 2.0 ** -10) == 0x02  # between 1 and 2 subnormal steps: even -> 2
    assert enc(15 * 2.0 ** -10) == 0x08  # between 7 * 2^-9 and 2^-6: even -> min normal
    assert enc(432.0) == 0x7E       # between 416 and 448: even mantissa -> 448
    assert enc(449.0) == 0x7E and enc(1e30) == 0x7E and enc(float("inf")) == 0x7E
    assert enc(-1e30) == 0xFE and enc(float("-inf")) == 0xFE
    assert enc(-0.0) == 0x80 and enc(0.0) == 0x00
    assert enc(-1e-6) == 0x80       # rounds to zero, keeps the sign


def test_e4m3_encode_monotone_and_roundtrip(oracle_mod):
    table = oracle_mod.e4m3_table()
    # every finite code round-trips
    for c in range(256):
        if not math.isnan(table[c]):
            assert oracle_mod.e4m3_encode(table[c]) == c or (table[c] == 0 and c in (0, 0x80))
    ys = np.linspace(0, 500, 20001).astype(np.float32)
    codes = [oracle_mod.e4m3_encode(float(y)) for y in ys]
    assert all(a <= b for a, b in zip(codes, codes[1:]))


# ----------------------------------------------------------- cache writes
def _tiny_pool(w):
    nbytes = 16 * w.n_kv_heads * w.head_dim * w.elem_bytes * w.num_blocks
    return np.zeros(nbytes, np.uint8), np.zeros(nbytes, np.uint8)


def test_reshape_places_each_token_in_its_slot(oracle_mod):
    w = W.make("tiny_fp16")
    kp, vp = _tiny_pool(w)
    kp[:] = 0xAB
    vp[:] = 0xCD
    for s in range(w.S):
        k, v = w.kv_bits(s, 0, int(w.ctx_lens[s]))
        slots = w.slots(s, 0, int(w.ctx_lens[s]))
        slots[3] = -1  # skipped token
        assert oracle_mod.reshape_and_cache("fp16", w.num_blocks, 16, w.n_kv_heads, w.head_dim,
                                            k, v, slots, 1.0, 1.0, kp, vp) == 0
    K = kp.view(np.uint16).reshape(w.num_blocks, w.n_kv_heads, 16, w.head_dim)
    V = vp.view(np.uint16).reshape(w.num_blocks, w.n_kv_heads, 16, w.head_dim)
    written = np.zeros(K.shape[0] * 16, bool)
    for s in range(w.S):
        n = int(w.ctx_lens[s])
        k, v = w.kv_bits(s, 0, n)
        for t in range(n):
            blk = w.block_tables[s, t // 16]
            if t == 3:
                assert np.all(K[blk, :, t % 16, :] == 0xABAB)
                continue
            assert np.array_equal(K[blk, :, t % 16, :], k[t])
            assert np.array_equal(V[blk, :, t % 16, :], v[t])
            written[blk * 16 + t % 16] = True
    # untouched slots keep their bytes
    flat = K.transpose(0, 2, 1, 3).reshape(-1, w.n_kv_heads * w.head_dim)
    assert np.all(flat[~written] == 0xABAB)


def test_reshape_out_of_range_slot_reports(oracle_mod):
    w = W.make("tiny_fp16")
    kp, vp = _tiny_pool(w)
    k, v = w.kv_bits(0, 0, 2)
    slots = np.array([0, w.num_blocks * 16], np.int64)
    assert oracle_mod.reshape_and_cache("fp16", w.num_blocks, 16, w.n_kv_heads, w.head_dim, k, v,
                                        slots, 1.0, 1.0, kp, vp) == -1


def test_reshape_fp8_codes_are_quantised_inputs(oracle_mod):
    """FP8 pool bytes equal the scalar quantiser applied to each written value."""
    w = W.make("llama3_8b_fp8", scale_down=32, steps=1)
    w.compute_fp8_scales()
    nbytes = 16 * w.n_kv_heads * w.head_dim * w.num_blocks
    kp, vp = np.zeros(nbytes, np.uint8), np.zeros(nbytes, np.uint8)
    s, n = 0, 20
    k, v = w.kv_bits(s, 0, n)
    slots = w.slots(s, 0, n)
    oracle_mod.reshape_and_cache("fp8_e4m3", w.num_blocks, 16, w.n_kv_heads, w.head_dim, k, v,
                                 slots, w.k_scale, w.v_scale, kp, vp)
    K = kp.reshape(w.num_blocks, w.n_kv_heads, 16, w.head_dim)
    xs = oracle_mod.value16("bf16", k[:, :2, :8])
    for t in range(n):
        blk = w.block_tables[s, t // 16]
        for h in range(2):
            for i in range(8):
                assert K[blk, h, t % 16, i] == oracle_mod.quantize_e4m3(xs[t, h, i], w.k_scale)


def test_copy_blocks(oracle_mod):
    w = W.make("tiny_fp16")
    kp, vp = _tiny_pool(w)
    rng = np.random.default_rng(3)
    kp[:] = rng.integers(0, 256, kp.size)
    vp[:] = rng.integers(0, 256, vp.size)
    K0 = kp.copy().reshape(w.num_blocks, -1)
    V0 = vp.copy().reshape(w.num_blocks, -1)
    pairs = np.array([[3, 9], [5, 0]], np.int32)
    assert oracle_mod.copy_blocks("fp16", w.num_blocks, 16, w.n_kv_heads, w.head_dim, pairs,
                                  kp, vp) == 0
    K, V = kp.reshape(w.num_blocks, -1), vp.reshape(w.num_blocks, -1)
    assert np.array_equal(K[9], K0[3]) and np.array_equal(V[0], V0[5])
    untouched = [b for b in range(w.num_blocks) if b not in (9, 0)]
    assert np.array_equal(K[untouched], K0[untouched])


# ------------------------------------------------------------- attention
def _fill_tiny(oracle_mod, w):
    kp, vp = _tiny_pool(w)
    for s in range(w.S):
        n = int(w.ctx_lens[s])
        k, v = w.kv_bits(s, 0, n)
        oracle_mod.reshape_and_cache("fp16", w.num_blocks, 16, w.n_kv_heads, w.head_dim, k, v,
                                     w.slots(s, 0, n), 1.0, 1.0, kp, vp)
    return kp, vp


def _attn(oracle_mod, w, kp, vp, q, tables=None, ctx=None, probs=False, kv_dtype=None,
          q_dtype=None, num_blocks=None, scale=None):
    return oracle_mod.paged_attention(
        kv_dtype or w.kv_dtype, q_dtype or w.in_dtype, num_blocks or w.num_blocks, 16,
        w.n_kv_heads, w.head_dim, kp, vp, w.k_scale, w.v_scale, q,
        w.block_tables if tables is None else tables, w.ctx_lens if ctx is None else ctx,
        w.softmax_scale if scale is None else scale, want_probs=probs)


def test_permutation_invariance_bit_exact(oracle_mod):
    """(2) Relabelling physical blocks (moving tile data and mapping the tables
    through the same permutation) leaves the output bit-identical."""
    w = W.make("tiny_fp16")
    kp, vp = _fill_tiny(oracle_mod, w)
    q = w.q_bits()
    out = _attn(oracle_mod, w, kp, vp, q)
    perm = np.random.default_rng(11).permutation(w.num_blocks)
    Kb, Vb = kp.reshape(w.num_blocks, -1), vp.reshape(w.num_blocks, -1)
    kp2, vp2 = np.empty_like(Kb), np.empty_like(Vb)
    kp2[perm] = Kb
    vp2[perm] = Vb
    tables2 = perm[w.block_tables].astype(np.int32)
    out2 = _attn(oracle_mod, w, kp2.ravel(), vp2.ravel(), q, tables=tables2)
    assert np.array_equal(out, out2)
    # and a wrong table (one entry swapped) does change it
    bad = w.block_tables.copy()
    bad[0, [0, 1]] = bad[0, [1, 0]]
    assert not np.array_equal(_attn(oracle_mod, w, kp, vp, q, tables=bad)[0], out[0])


def test_slab_identity(oracle_mod):
    """(3) Consecutive block ids, laid out contiguously, give the same result as
    attention over a contiguous [ctx, Hkv, d] slab."""
    w = W.make("tiny_fp16")
    S, Hkv, d = w.S, w.n_kv_heads, w.head_dim
    max_ctx = int(w.ctx_lens.max())
    tables = np.zeros_like(w.block_tables)
    nxt = 0
    kp, vp = _tiny_pool(w)
    Kslab = np.zeros((S, max_ctx, Hkv, d))
    Vslab = np.zeros((S, max_ctx, Hkv, d))
    for s in range(S):
        n = int(w.ctx_lens[s])
        nb = -(-n // 16)
        tables[s, :nb] = np.arange(nxt, nxt + nb)
        nxt += nb
        k, v = w.kv_bits(s, 0, n)
        Kslab[s, :n] = k.view(np.float16).astype(np.float64)
        Vslab[s, :n] = v.view(np.float16).astype(np.float64)
        slots = (tables[s, np.arange(n) // 16].astype(np.int64) * 16 + np.arange(n) % 16)
        oracle_mod.reshape_and_cache("fp16", w.num_blocks, 16, Hkv, d, k, v, slots, 1, 1, kp, vp)
    q = w.q_bits()
    paged = _attn(oracle_mod, w, kp, vp, q, tables=tables)
    slab = oracle_mod.slab_attention(Kslab, Vslab, q.view(np.float16).astype(np.float64),
                                     w.ctx_lens, w.softmax_scale)
    assert np.array_equal(paged, slab)


def _single_seq(n, Hq=4, Hkv=2, d=64, dtype="fp16"):
    nb = max(1, -(-n // 16))
    w = W.Workload(name="hand", index=0, kv_dtype=dtype, n_q_heads=Hq, n_kv_heads=Hkv,
                   head_dim=d, ctx_lens=np.array([n], np.int32), num_blocks=nb + 3,
                   block_tables=np.array([list(range(nb + 2, 2, -1))[:nb]], np.int32))
    return w


def _write(oracle_mod, w, kvals, vvals, kp=None, vp=None):
    """kvals/vvals: float arrays [n, Hkv, d] exactly representable in fp16."""
    if kp is None:
        kp, vp = _tiny_pool(w)
    n = kvals.shape[0]
    k = kvals.astype(np.float16).view(np.uint16)
    v = vvals.astype(np.float16).view(np.uint16)
    oracle_mod.reshape_and_cache("fp16", w.num_blocks, 16, w.n_kv_heads, w.head_dim, k, v,
                                 w.slots(0, 0, n), 1.0, 1.0, kp, vp)
    return kp, vp


def _q(w, vals):
    return np.asarray(vals, np.float16).reshape(1, w.n_q_heads, w.head_dim).view(np.uint16)


def test_brute_force_ctx1_returns_v0(oracle_mod):
    """(4) One token: softmax weight 1, output equals that token's value."""
    w = _single_seq(1)
    rng = np.random.default_rng(1)
    kv = rng.standard_normal((2, 1, 2, 64)).astype(np.float16).astype(np.float64)
    kp, vp = _write(oracle_mod, w, kv[0], kv[1])
    q = _q(w, rng.standard_normal(4 * 64))
    out = _attn(oracle_mod, w, kp, vp, q)
    for g in range(4):
        assert np.array_equal(out[0, g], kv[1][0, g // 2])


def test_brute_force_equal_keys_and_zero_query_give_mean(oracle_mod):
    """(4) Equal logits -> uniform weights -> the mean of V, across a block
    boundary and a ragged tail (ctx 37)."""
    n = 37
    w = _single_seq(n)
    rng = np.random.default_rng(2)
    K = np.broadcast_to(rng.standard_normal((1, 2, 64)), (n, 2, 64)).astype(np.float16)
    V = np.zeros((n, 2, 64))
    V[:, 0, :] = np.arange(n)[:, None]        # kv head 0: value t in every dim
    V[:, 1, :] = -2.0 * np.arange(n)[:, None]  # kv head 1: -2t
    kp, vp = _write(oracle_mod, w, K.astype(np.float64), V)
    q = _q(w, rng.standard_normal(4 * 64))
    out = _attn(oracle_mod, w, kp, vp, q)
    mean_t = (n - 1) / 2.0
    for g in range(4):  # query heads 0,1 -> kv head 0; 2,3 -> kv head 1
        expect = mean_t if g < 2 else -2.0 * mean_t
        assert np.allclose(out[0, g], expect, rtol=0, atol=1e-12)
    # zero query, arbitrary keys: also the mean
    K2 = rng.standard_normal((n, 2, 64))
    kp, vp = _write(oracle_mod, w, K2, V)
    out0 = _attn(oracle_mod, w, kp, vp, _q(w, np.zeros(4 * 64)))
    assert np.allclose(out0[0, :2], mean_t, atol=1e-12)
    assert np.allclose(out0[0, 2:], -2.0 * mean_t, atol=1e-12)


def test_brute_force_dominant_key_selects_its_value(oracle_mod):
    """(4) One logit 64 above the rest: weight 1 - O(e^-64) on that token."""
    n, hot = 50, 33
    w = _single_seq(n)
    K = np.zeros((n, 2, 64))
    K[hot, :, 0] = 64.0
    V = np.random.default_rng(3).standard_normal((n, 2, 64)).astype(np.float16)
    kp, vp = _write(oracle_mod, w, K, V.astype(np.float64))
    qv = np.zeros((4, 64))
    qv[:, 0] = 8.0  # z_hot = 8 * 64 / sqrt(64) = 64, others 0
    out = _attn(oracle_mod, w, kp, vp, _q(w, qv))
    for g in range(4):
        assert np.allclose(out[0, g], V[hot, g // 2].astype(np.float64), atol=1e-12)


def test_huge_logits_shift_invariance(oracle_mod):
    """Softmax is invariant to a common shift of the logits; with logits in
    the thousands the result must still be finite and equal the shifted case."""
    n, hot = 40, 17
    w = _single_seq(n, Hq=2, Hkv=1, d=64)
    K = np.zeros((n, 1, 64))
    K[:, 0, 0] = 256.0
    K[hot, 0, 1] = 8.0
    V = np.random.default_rng(5).standard_normal((n, 1, 64)).astype(np.float16)
    kp, vp = _write(oracle_mod, w, K, V.astype(np.float64))
    qv = np.zeros((2, 64))
    qv[:, 0] = 256.0   # common logit 256 * 256 / 8 = 8192 for every token
    qv[:, 1] = 1.0     # plus 1 for the hot token
    out = _attn(oracle_mod, w, kp, vp, _q(w, qv))
    qv[:, 0] = 0.0     # same differences, no common shift
    ref = _attn(oracle_mod, w, kp, vp, _q(w, qv))
    assert np.all(np.isfinite(out))
    assert np.allclose(out, ref, atol=1e-12)


def test_brute_force_two_tokens_logistic(oracle_mod):
    """(4) Two tokens with logits 0 and ln 3 get weights 1/4 and 3/4."""
    w = _single_seq(2, Hq=1, Hkv=1, d=64)
    K = np.zeros((2, 1, 64))
    K[1, 0, 0] = 1.0
    V = np.zeros((2, 1, 64))
    V[0, 0, :] = 1.0
    V[1, 0, :] = 5.0
    kp, vp = _write(oracle_mod, w, K, V)
    qv = np.zeros((1, 64))
    qv[0, 0] = 1.0
    out = oracle_mod.paged_attention("fp16", "fp16", w.num_blocks, 16, 1, 64, kp, vp, 1.0, 1.0,
                                     _q(w, qv), w.block_tables, w.ctx_lens, math.log(3.0))
    assert np.allclose(out[0, 0], 0.25 * 1.0 + 0.75 * 5.0, atol=1e-13)


def test_softmax_rows_sum_to_one_and_unit_values(oracle_mod):
    """(5) Probabilities are a distribution; V == 1 gives output 1 exactly-ish."""
    w = W.make("tiny_fp16")
    kp, vp = _fill_tiny(oracle_mod, w)
    out, probs = _attn(oracle_mod, w, kp, vp, w.q_bits(), probs=True)
    for s in range(w.S):
        n = int(w.ctx_lens[s])
        p = probs[s, :, :n]
        assert np.all(p >= 0)
        assert np.allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        assert np.all(probs[s, :, n:] == 0)
    ones = np.full(vp.size // 2, 0x3C00, np.uint16).view(np.uint8)  # fp16 1.0 everywhere
    out1 = _attn(oracle_mod, w, kp, ones.copy(), w.q_bits())
    assert np.allclose(out1, 1.0, rtol=0, atol=1e-12)


def test_fp8_dequantisation_scales_values(oracle_mod):
    """A constant FP8 value code c with scale s reads back as decode(c) * s."""
    w = _single_seq(20, dtype="fp8_e4m3")
    w.k_scale, w.v_scale = 0.5, 0.25
    nbytes = 16 * w.n_kv_heads * w.head_dim * w.num_blocks
    kp = np.full(nbytes, 0x38, np.uint8)   # 1.0 -> 0.5 after scale
    vp = np.full(nbytes, 0x4C, np.uint8)   # E=9, M=4: 1.5 * 4 = 6 -> 1.5 after scale
    q = np.random.default_rng(4).standard_normal((1, 4, 64)).astype(np.float32)
    qb = W.f32_to_bf16_bits(q)
    out = oracle_mod.paged_attention("fp8_e4m3", "bf16", w.num_blocks, 16, 2, 64, kp, vp, 0.5,
                                     0.25, qb, w.block_tables, w.ctx_lens, w.softmax_scale)
    assert np.allclose(out, 1.5, atol=1e-12)


def test_zero_context_gives_zero_output(oracle_mod):
    w = W.make("tiny_fp16")
    kp, vp = _fill_tiny(oracle_mod, w)
    ctx = w.ctx_lens.copy()
    ctx[1] = 0
    out = _attn(oracle_mod, w, kp, vp, w.q_bits(), ctx=ctx)
    assert np.all(out[1] == 0)
    assert np.any(out[0] != 0)


def test_invalid_table_entry_rejected(oracle_mod):
    w = W.make("tiny_fp16")
    kp, vp = _fill_tiny(oracle_mod, w)
    bad = w.block_tables.copy()
    bad[2, 0] = w.num_blocks
    with pytest.raises(ValueError):
        _attn(oracle_mod, w, kp, vp, w.q_bits(), tables=bad)
