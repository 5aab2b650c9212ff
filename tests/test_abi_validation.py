"""Argument checks of the device entry points declared in include/pa.h, on the
host.  Every case below is rejected (or, for empty work, accepted) before the
library makes any CUDA call, so the pools' regions and the tensors' addresses
are fake ones that nothing dereferences; where a GPU is present the file skips
itself rather than hand those addresses to a device."""
import math

import pytest
import torch

N = pytest.importorskip("paged_kv_cache_270_gb300._native")

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="host-only checks with fake device addresses")

FAKE_K, FAKE_V = 1 << 40, 1 << 41
A = 1 << 44  # a 16-byte-aligned fake device address for q, out, tables and lengths


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_270_gb300 import build
    build.build()
    return N.lib()


@pytest.fixture
def pool(lib):  # 2 layers, 64 blocks, 2 KV heads of 64 dims, binary16
    h = N.pa_pool_create(N.make_desc(2, 64, 2, 64, N.PA_FP16), FAKE_K, FAKE_V)
    yield h
    N.pa_pool_destroy(h)


def _code(fn, *args, **kw):
    with pytest.raises(N.PAError) as e:
        fn(*args, **kw)
    return e.value.code


INV, UNS = N.PA_ERR_INVALID, N.PA_ERR_UNSUPPORTED


def _decode(pool, **kw):
    a = dict(layer=0, out=A, out_dtype=N.PA_FP16, q=A, tables=A, max_blocks=4, ctx=A, S=3,
             Hq=4, scale=0.125, num_splits=1, ws=0, ws_bytes=0)
    a.update(kw)
    N.pa_decode(pool, a["layer"], a["out"], a["out_dtype"], a["q"], a["tables"], a["max_blocks"],
                a["ctx"], a["S"], a["Hq"], a["scale"], a["num_splits"], a["ws"], a["ws_bytes"], 0)


@pytest.mark.parametrize("kw, code", [
    (dict(layer=2), INV), (dict(layer=-1), INV),
    (dict(Hq=3), INV),                         # not a multiple of the 2 KV heads
    (dict(Hq=18), UNS),                        # 9 query heads per KV head
    (dict(S=70000), UNS), (dict(S=-1), INV), (dict(max_blocks=0), INV),
    (dict(out_dtype=N.PA_BF16), INV),          # neither the query dtype nor fp32
    (dict(scale=math.nan), INV), (dict(scale=math.inf), INV),
    (dict(out=0), INV), (dict(q=A + 8), INV),  # null, misaligned
    (dict(num_splits=-2), INV),
    (dict(num_splits=2), INV),                 # two splits need a workspace
    (dict(num_splits=2, ws=A, ws_bytes=16), INV),
])
def test_decode_rejects(pool, kw, code):
    assert _code(_decode, pool, **kw) == code


def _decode_no_alloc(pool, **kw):
    a = dict(layer=0, out=A, out_dtype=N.PA_FP16, q=A, tables=A, max_blocks=4, ctx=A, S=3,
             Hq=4, scale=0.125, num_splits=1)
    a.update(kw)
    N.pa_decode_no_alloc(pool, a["layer"], a["out"], a["out_dtype"], a["q"], a["tables"],
                         a["max_blocks"], a["ctx"], a["S"], a["Hq"], a["scale"], a["num_splits"], 0)


@pytest.mark.parametrize("kw, code", [
    (dict(layer=2), INV), (dict(Hq=3), INV), (dict(Hq=18), UNS), (dict(S=70000), UNS),
    (dict(S=-1), INV), (dict(max_blocks=0), INV), (dict(out_dtype=N.PA_BF16), INV),
    (dict(scale=math.nan), INV), (dict(out=0), INV), (dict(q=A + 8), INV),
    (dict(num_splits=-2), INV),
    # an empty batch is still checked for its output type and scale, as pa_decode does
    (dict(S=0, out_dtype=N.PA_BF16), INV), (dict(S=0, scale=math.inf), INV),
])
def test_decode_no_alloc_checks_match_decode(pool, kw, code):
    assert _code(_decode, pool, **kw) == code
    assert _code(_decode_no_alloc, pool, **kw) == code


def test_decode_empty_batch_is_accepted(pool):
    _decode(pool, S=0)
    _decode(pool, S=0, out=0, q=0)  # nothing is read or written
    _decode_no_alloc(pool, S=0, out=0, q=0)


@pytest.mark.parametrize("B, s, splits", [(10, 1, 1), (10, 3, 3), (10, 4, 4), (10, 6, 5),
                                          (10, 10, 10), (10, 99, 10), (1, 5, 1)])
def test_workspace_bytes_closed_form(pool, B, s, splits):
    """s requested splits of B pages run as ceil(B / ceil(B / s)) splits of
    ceil(B / s) pages; each keeps (m, l, o[d]) in fp32 per (sequence, query head)."""
    S, Hq, d = 3, 4, 64
    want = S * Hq * splits * (d + 2) * 4 if splits > 1 else 0
    assert N.pa_decode_workspace_bytes(pool, S, Hq, B, s) == want


def test_decode_no_alloc_rejects_oversized_explicit_splits(pool):
    S, Hq = 4000, 4
    row = S * Hq * (64 + 2) * 4      # one split's partials
    assert 2 * row > (8 << 20)       # above PA_NOALLOC_SCRATCH_BYTES
    code = _code(N.pa_decode_no_alloc, pool, 0, A, N.PA_FP16, A, A, 8, A, S, Hq, 0.125, 2, 0)
    assert code == INV


def _prefill(pool, **kw):
    a = dict(layer=0, out=A, out_dtype=N.PA_FP16, q=A, q_start=A, tables=A, max_blocks=4, ctx=A,
             S=2, Hq=4, max_chunk=32, scale=0.125)
    a.update(kw)
    N.pa_prefill(pool, a["layer"], a["out"], a["out_dtype"], a["q"], a["q_start"], a["tables"],
                 a["max_blocks"], a["ctx"], a["S"], a["Hq"], a["max_chunk"], a["scale"], 0)


@pytest.mark.parametrize("kw, code", [
    (dict(layer=2), INV), (dict(S=-1), INV), (dict(max_blocks=0), INV),
    (dict(Hq=3), INV), (dict(Hq=18), UNS), (dict(max_chunk=-1), INV),
    (dict(out_dtype=N.PA_BF16), INV), (dict(scale=math.nan), INV),
    (dict(S=70000), UNS), (dict(out=0), INV), (dict(q_start=0), INV), (dict(q=A + 4), INV),
])
def test_prefill_rejects(pool, kw, code):
    assert _code(_prefill, pool, **kw) == code


def test_prefill_empty_work_is_accepted(pool):
    _prefill(pool, S=0)
    _prefill(pool, max_chunk=0, out=0, q=0)


@pytest.mark.parametrize("args, code", [
    ((5, A, A, A, 4), INV), ((0, A, A, A, -1), INV),   # layer, T
    ((0, 0, A, A, 4), INV), ((0, A, A, 0, 4), INV),    # null k, null slot mapping
    ((0, A + 2, A, A, 4), INV),                        # misaligned k
])
def test_reshape_and_cache_rejects(pool, args, code):
    assert _code(N.pa_reshape_and_cache, pool, *args, 0) == code


def test_reshape_and_cache_no_tokens(pool):
    N.pa_reshape_and_cache(pool, 1, 0, 0, 0, 0, 0)


@pytest.mark.parametrize("args, code", [
    ((-1, A, 1), INV), ((0, A, -1), INV), ((0, 0, 1), INV), ((0, A, 70000), UNS),
])
def test_copy_blocks_rejects(pool, args, code):
    assert _code(N.pa_copy_blocks, pool, *args, 0) == code


def test_copy_blocks_no_pairs(pool):
    N.pa_copy_blocks(pool, 1, 0, 0, 0)


@pytest.mark.parametrize("fn", [N.pa_swap_out, N.pa_swap_in])
def test_swap_rejects_and_accepts_nothing(pool, fn):
    assert _code(fn, pool, -1, A, A, 0) == INV
    assert _code(fn, pool, 3, 0, A, 0) == INV
    assert _code(fn, pool, 3, A, 0, 0) == INV
    fn(pool, 0, 0, 0, 0)


def test_swap_record_sizes(lib):
    # one block's record: K and V tiles of every layer and KV head (16 x d x bytes each),
    # plus, for block-scaled pools, their fp32 scales rounded up to 16 bytes
    h = N.pa_pool_create(N.make_desc(2, 64, 2, 64, N.PA_FP16), FAKE_K, FAKE_V)
    assert N.pa_swap_block_bytes(h) == 2 * 2 * 2 * 16 * 64 * 2
    N.pa_pool_destroy(h)
    h = N.pa_pool_create(N.make_desc(1, 64, 8, 128, N.PA_FP8_E4M3_BLOCK), FAKE_K, FAKE_V)
    assert N.pa_swap_block_bytes(h) == 2 * 1 * 8 * 16 * 128 + 64
    N.pa_pool_destroy(h)
    h = N.pa_pool_create(N.make_desc(3, 64, 1, 64, N.PA_FP8_E4M3_BLOCK), FAKE_K, FAKE_V)
    assert N.pa_swap_block_bytes(h) == 2 * 3 * 1 * 16 * 64 + 32  # 24 bytes of scales -> 32
    N.pa_pool_destroy(h)
