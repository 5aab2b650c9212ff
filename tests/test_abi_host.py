"""The C-ABI library on the host (no GPU): it loads, exports every entry point
include/pa.h declares, sizes pools by the closed form, and its block allocator
matches the reference model table for table and refcount for refcount."""
import os
import random
import re

import numpy as np
import pytest

from conftest import ROOT
from oracle.allocator_model import AllocatorModel, InvalidRequest, OutOfBlocks

N = pytest.importorskip("paged_kv_cache_270_gb300._native")

FAKE_K, FAKE_V = 1 << 40, 1 << 41  # device addresses the host code never dereferences


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_270_gb300 import build
    build.build()
    return N.lib()


def _declared_symbols():
    syms = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            syms += re.findall(r"PA_API\s+int\s+(pa_\w+)\s*\(", open(os.path.join(inc, f)).read())
    return syms


def test_library_exports_every_declared_symbol(lib):
    syms = _declared_symbols()
    assert len(syms) >= 19
    for s in syms:
        assert hasattr(lib, s), s
    bound = {name for name, _ in N._SIGS}
    assert bound == set(syms), "binding and header disagree"


def test_bytes_per_token_closed_form(lib):
    assert N.pa_kv_bytes_per_token(80, 8, 128, N.PA_FP16) == 327680
    assert N.pa_kv_bytes_per_token(80, 8, 128, N.PA_BF16) == 327680
    assert N.pa_kv_bytes_per_token(80, 8, 128, N.PA_FP8_E4M3) == 163840
    with pytest.raises(N.PAError):
        N.pa_kv_bytes_per_token(80, 8, 128, N.PA_FP32)


@pytest.mark.parametrize("layers,heads,d,dt", [(1, 2, 64, N.PA_FP16), (1, 8, 128, N.PA_BF16),
                                               (80, 8, 128, N.PA_FP8_E4M3),
                                               (32, 8, 128, N.PA_BF16)])
def test_pool_bytes_and_budget(lib, layers, heads, d, dt):
    desc = N.make_desc(layers, 100, heads, d, dt, 0.5, 0.5)
    kb, vb = N.pa_pool_bytes(desc)
    per_tok = N.pa_kv_bytes_per_token(layers, heads, d, dt)
    assert kb == vb and kb + vb == per_tok * 100 * 16
    per_block = per_tok * 16
    assert N.pa_pool_blocks_for_budget(desc, per_block * 7 + per_block - 1) == 7
    with pytest.raises(N.PAError) as e:
        N.pa_pool_blocks_for_budget(desc, per_block - 1)
    assert e.value.code == N.PA_ERR_NO_MEMORY


@pytest.mark.parametrize("layers,heads,nb", [(1, 2, 7), (80, 8, 100), (3, 1, 5)])
def test_block_scaled_pool_sizes(lib, layers, heads, nb):
    """Block-scaled FP8: the tiles as for FP8, plus one fp32 scale per (layer,
    block, kv head) at the end of each region, rounded up to 16 bytes; the
    swap record carries the block's 2 * layers * heads scales, padded."""
    d = 128
    desc = N.make_desc(layers, nb, heads, d, N.PA_FP8_E4M3_BLOCK)
    kb, vb = N.pa_pool_bytes(desc)
    tiles = layers * nb * heads * 16 * d
    table = -(-(layers * nb * heads * 4) // 16) * 16
    assert kb == vb == tiles + table
    assert N.pa_kv_bytes_per_token(layers, heads, d, N.PA_FP8_E4M3_BLOCK) == 2 * layers * heads * d
    per_block = 2 * layers * heads * (16 * d + 4)
    n = N.pa_pool_blocks_for_budget(desc, per_block * 9 + 64)
    desc9 = N.make_desc(layers, n, heads, d, N.PA_FP8_E4M3_BLOCK)
    assert sum(N.pa_pool_bytes(desc9)) <= per_block * 9 + 64
    assert n in (8, 9)
    h = N.pa_pool_create(desc, FAKE_K, FAKE_V)
    try:
        rec = N.pa_swap_block_bytes(h)
        assert rec == 2 * layers * heads * 16 * d + -(-(2 * layers * heads * 4) // 16) * 16
    finally:
        N.pa_pool_destroy(h)


def test_invalid_descriptions(lib):
    bad = [N.make_desc(1, 10, 2, 96, N.PA_FP16),            # head_dim
           N.make_desc(1, 10, 2, 64, N.PA_FP16, block_size=32),
           N.make_desc(1, 10, 2, 64, N.PA_FP8_E4M3, 0.0, 1.0),  # scale
           N.make_desc(1, 10, 2, 64, N.PA_FP8_E4M3, float("inf"), 1.0),
           N.make_desc(0, 10, 2, 64, N.PA_FP16),
           N.make_desc(1, 10, 0, 64, N.PA_FP16),
           N.make_desc(1, 10, 2, 64, 7)]
    for d in bad:
        with pytest.raises(N.PAError):
            N.pa_pool_create(d, FAKE_K, FAKE_V)
    with pytest.raises(N.PAError) as e:
        N.pa_pool_create(N.make_desc(1, 0, 2, 64, N.PA_FP16), FAKE_K, FAKE_V)
    assert e.value.code == N.PA_ERR_NO_MEMORY
    with pytest.raises(N.PAError):  # misaligned region
        N.pa_pool_create(N.make_desc(1, 4, 2, 64, N.PA_FP16), FAKE_K + 8, FAKE_V)


@pytest.fixture
def pool(lib):
    h = N.pa_pool_create(N.make_desc(1, 64, 2, 64, N.PA_FP16), FAKE_K, FAKE_V)
    yield h
    N.pa_pool_destroy(h)


def test_allocator_matches_model_on_random_operations(pool):
    rnd = random.Random(5)
    m = AllocatorModel(64)
    live = []
    for step in range(3000):
        op = rnd.random()
        if op < 0.4:
            n = rnd.randint(0, 9)
            try:
                want = m.alloc(n)
            except OutOfBlocks:
                with pytest.raises(N.PAError) as e:
                    N.pa_block_alloc(pool, n)
                assert e.value.code == N.PA_ERR_OUT_OF_BLOCKS
                continue
            got = N.pa_block_alloc(pool, n)
            assert list(got) == want
            live.append(want)
        elif op < 0.7 and live:
            t = live.pop(rnd.randrange(len(live)))
            m.free(t)
            N.pa_block_free(pool, t)
        elif op < 0.85 and live:
            t = rnd.choice(live)[:3]
            m.incref(t)
            N.pa_block_incref(pool, t)
            live.append(list(t))
        elif op < 0.93:
            # an invalid request: double free or incref of a free block
            bad = [rnd.randrange(64)] * rnd.randint(1, 3)
            try:
                m.free(bad)
                live_flat = [b for tt in live for b in tt]
                # model accepted: only if the refs exist; mirror it and drop them from live
                N.pa_block_free(pool, bad)
                for b in bad:
                    for tt in live:
                        if b in tt:
                            tt.remove(b)
                            break
                del live_flat
            except InvalidRequest:
                with pytest.raises(N.PAError) as e:
                    N.pa_block_free(pool, bad)
                assert e.value.code == N.PA_ERR_INVALID
        else:
            b = rnd.randrange(64)
            assert N.pa_block_refcount(pool, b) == m.refcount[b]
        assert N.pa_pool_stats(pool) == m.stats()
    assert [N.pa_block_refcount(pool, b) for b in range(64)] == m.refcount


def test_cow_best_of_8_matches_model(pool, lib):
    h = N.pa_pool_create(N.make_desc(1, 1024, 8, 128, N.PA_BF16), FAKE_K, FAKE_V)
    try:
        m = AllocatorModel(1024)
        prompt = N.pa_block_alloc(h, 126)   # 2008 tokens
        assert list(prompt) == m.alloc(126)
        tables, mtables = [], []
        for b in range(8):
            if b:
                N.pa_block_incref(h, prompt)
                m.incref(list(prompt))
            tables.append(np.concatenate([prompt, np.zeros(4, np.int32)]).astype(np.int32))
            mtables.append(list(prompt) + [0] * 4)
        pairs = []
        for b in range(8):
            got = N.pa_cow_prepare(h, tables[b], 2008)
            want = m.cow_prepare(mtables[b], 2008)
            assert got == want
            assert list(tables[b]) == mtables[b]
            if got:
                pairs.append(got)
        assert len(pairs) == 7
        assert N.pa_block_refcount(h, int(prompt[-1])) == 1
        for b in range(8):
            for j in range(4):
                blk = N.pa_block_alloc(h, 1)
                tables[b][126 + j] = blk[0]
                mtables[b][126 + j] = m.alloc(1)[0]
            assert list(tables[b]) == mtables[b]
        assert N.pa_pool_stats(h) == m.stats() == (165, 1024 - 165, 125)
        assert [N.pa_block_refcount(h, b) for b in range(1024)] == m.refcount
        # cancellation returns everything
        for t in tables:
            N.pa_block_free(h, t)
        assert N.pa_pool_stats(h) == (0, 1024, 0)
    finally:
        N.pa_pool_destroy(h)


def test_cow_edge_cases(pool):
    ids = N.pa_block_alloc(pool, 2)
    row = ids.copy()
    assert N.pa_cow_prepare(pool, row, 16) is None          # opens a new block
    assert N.pa_cow_prepare(pool, row, 5) is None           # sole owner
    N.pa_block_incref(pool, ids[:1])
    assert N.pa_cow_prepare(pool, row, 5) == (ids[0], 2)
    assert row[0] == 2 and N.pa_block_refcount(pool, int(ids[0])) == 1
    # out of blocks: no change
    rest = N.pa_block_alloc(pool, N.pa_pool_stats(pool)[1])
    N.pa_block_incref(pool, row[:1])
    before = row.copy()
    with pytest.raises(N.PAError) as e:
        N.pa_cow_prepare(pool, row, 3)
    assert e.value.code == N.PA_ERR_OUT_OF_BLOCKS
    assert np.array_equal(row, before) and N.pa_block_refcount(pool, int(row[0])) == 2
    N.pa_block_free(pool, rest)


def test_last_error_message(pool):
    with pytest.raises(N.PAError) as e:
        N.pa_block_free(pool, [3])
    assert "double free" in str(e.value) or "below refcount" in str(e.value)
    assert "double free" in N.last_error()


def test_rows_per_layer_limit(lib):
    """A layer holds at most 2^31 - 1 token rows (blocks x KV heads x 16), the
    range of the kernels' 32-bit tile coordinates: sizing, budget and creation
    agree on the boundary."""
    heads = 64
    top = (2**31 - 1) // (heads * 16)                  # 2,097,151 blocks
    ok = N.make_desc(1, top, heads, 64, N.PA_FP8_E4M3, 1.0, 1.0)
    over = N.make_desc(1, top + 1, heads, 64, N.PA_FP8_E4M3, 1.0, 1.0)
    kb, _ = N.pa_pool_bytes(ok)
    assert kb == top * heads * 16 * 64
    with pytest.raises(N.PAError) as e:
        N.pa_pool_bytes(over)
    assert e.value.code == N.PA_ERR_UNSUPPORTED
    with pytest.raises(N.PAError) as e:
        N.pa_pool_create(over, FAKE_K, FAKE_V)
    assert e.value.code == N.PA_ERR_UNSUPPORTED
    h = N.pa_pool_create(ok, FAKE_K, FAKE_V)
    N.pa_pool_destroy(h)
    assert N.pa_pool_blocks_for_budget(ok, 1 << 50) == top
    assert N.pa_pool_blocks_for_budget(ok, 2 * kb) == top
    assert N.pa_pool_blocks_for_budget(ok, 2 * kb - 1) == top - 1


def _c_kind(param: str):
    param = param.strip()
    if "*" in param:
        return "ptr"
    ctype = param.rsplit(None, 1)[0].replace("const", "").strip()
    return {"int": ("int", 4), "int32_t": ("int", 4), "size_t": ("int", 8),
            "uint64_t": ("int", 8), "float": ("float", 4)}[ctype]


def _py_kind(t):
    import ctypes
    if t in (ctypes.c_void_p, ctypes.c_char_p) or hasattr(t, "_type_") and issubclass(
            t, ctypes._Pointer):
        return "ptr"
    if t is ctypes.c_float:
        return ("float", 4)
    return ("int", ctypes.sizeof(t))


def test_binding_signatures_match_header(lib):
    """Every entry point's argument list in the ctypes binding has the header's
    arity and, position by position, the same kind (pointer, 32- or 64-bit
    integer, float): a mismatch would pass garbage across the ABI."""
    decls = {}
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            for name, params in re.findall(r"PA_API\s+int\s+(pa_\w+)\s*\(([^)]*)\)\s*;", text):
                decls[name] = [_c_kind(p) for p in params.split(",")]
    sigs = dict(N._SIGS)
    assert set(sigs) == set(decls)
    for name, kinds in decls.items():
        assert [_py_kind(t) for t in sigs[name]] == kinds, name
