"""Prefix caching by block hash, host side: the hash is pinned to published
FNV-1a test vectors, the library's chain hashes and cache policy match the
reference model exactly, and a shared system prompt is served from the cache
(the page's >99% hit rate for a chat service's system prompt)."""
import random

import numpy as np
import pytest

from oracle.allocator_model import AllocatorModel, fnv1a64, prefix_chain_hashes

N = pytest.importorskip("paged_kv_cache_270_gb300._native")
FAKE_K, FAKE_V = 1 << 40, 1 << 41


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_270_gb300 import build
    build.build()
    return N.lib()


def test_fnv1a64_published_vectors():
    # Fowler/Noll/Vo reference test vectors for 64-bit FNV-1a
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_chain_hashes_match_model(lib):
    rng = np.random.default_rng(1)
    for n in (0, 15, 16, 17, 100, 2048):
        toks = rng.integers(-2**31, 2**31 - 1, n, dtype=np.int64).astype(np.int32)
        for parent in (0, 0x123456789ABCDEF0):
            got = N.pa_prefix_hash(toks, parent)
            want = prefix_chain_hashes(list(toks), parent)
            assert [int(x) for x in got] == want
    # a chain depends on every earlier block
    a = np.arange(64, dtype=np.int32)
    b = a.copy()
    b[3] += 1
    ha, hb = N.pa_prefix_hash(a), N.pa_prefix_hash(b)
    assert all(x != y for x, y in zip(ha, hb))


def test_prefix_cache_matches_model_on_random_operations(lib):
    h = N.pa_pool_create(N.make_desc(1, 96, 2, 64, N.PA_FP16), FAKE_K, FAKE_V)
    m = AllocatorModel(96)
    rnd = random.Random(11)
    prompts = [list(np.random.default_rng(i).integers(0, 50000, 16 * rnd.randint(1, 8)))
               for i in range(6)]
    live = []  # (table of ids)
    try:
        for step in range(1500):
            op = rnd.random()
            if op < 0.35:
                p = rnd.choice(prompts)
                hashes = prefix_chain_hashes(p)
                got = list(N.pa_prefix_lookup(h, np.array(hashes, np.uint64)))
                want = m.prefix_lookup(hashes)
                assert got == want
                need = len(hashes) - len(got)
                if need > len(m.free_stack):
                    if got:
                        N.pa_block_free(h, got)
                        m.free(got)
                    continue
                new = list(N.pa_block_alloc(h, need))
                assert new == m.alloc(need)
                table = got + new
                N.pa_prefix_register(h, np.array(hashes[len(got):], np.uint64),
                                     np.array(new, np.int32))
                m.prefix_register(hashes[len(got):], new)
                live.append(table)
            elif op < 0.7 and live:
                t = live.pop(rnd.randrange(len(live)))
                N.pa_block_free(h, t)
                m.free(t)
            else:
                k = rnd.randint(0, 8)
                assert N.pa_prefix_evict(h, k) == m.prefix_evict(k)
            assert N.pa_pool_stats(h) == m.stats()
            assert N.pa_prefix_stats(h) == (len(m.prefix), m.lookups, m.hits)
        assert [N.pa_block_refcount(h, b) for b in range(96)] == m.refcount
    finally:
        N.pa_pool_destroy(h)


def test_shared_system_prompt_hit_rate(lib):
    """'Capítulo 8 ...', section 8.3: over 99% of a chat service's system-prompt
    blocks come from the cache."""
    h = N.pa_pool_create(N.make_desc(1, 8192, 8, 128, N.PA_BF16), FAKE_K, FAKE_V)
    try:
        system = np.random.default_rng(0).integers(0, 128000, 2048).astype(np.int32)
        hs = N.pa_prefix_hash(system)
        assert len(hs) == 128
        tables = []
        for r in range(120):
            hit = N.pa_prefix_lookup(h, hs)
            own = N.pa_block_alloc(h, len(hs) - len(hit))
            if len(own):
                N.pa_prefix_register(h, hs[len(hit):], own)
            tables.append(np.concatenate([hit, own]))
        entries, lookups, hits = N.pa_prefix_stats(h)
        assert entries == 128 and lookups == 120 * 128
        assert hits / lookups > 0.99
        assert all(np.array_equal(t, tables[0]) for t in tables)
        assert N.pa_block_refcount(h, int(tables[0][0])) == 121  # 120 requests + cache
        for t in tables:
            N.pa_block_free(h, t)
        assert N.pa_pool_stats(h)[0] == 128          # still cached
        assert N.pa_prefix_evict(h, 1000) == 128
        assert N.pa_pool_stats(h) == (0, 8192, 0)
    finally:
        N.pa_pool_destroy(h)


def test_register_rejects_free_block(lib):
    h = N.pa_pool_create(N.make_desc(1, 8, 2, 64, N.PA_FP16), FAKE_K, FAKE_V)
    try:
        with pytest.raises(N.PAError):
            N.pa_prefix_register(h, np.array([5], np.uint64), np.array([3], np.int32))
        assert N.pa_prefix_stats(h)[0] == 0
    finally:
        N.pa_pool_destroy(h)
