"""Pins of the allocator reference model against the pages' printed numbers
and the block-manager invariants (no GPU)."""
import random

import pytest

from conftest import golden_lines
from oracle.allocator_model import (AllocatorModel, InvalidRequest, OutOfBlocks, blocks_for,
                                    internal_waste, slot_of)


def _golden_dict(name):
    return {k: v for k, v in golden_lines(name)}


def test_figure_block_table_slots():
    """'PagedAttention y Gestión de KV-Cache', section 2 figure."""
    rows = golden_lines("block_table_figure.txt")
    table = [int(p) for kind, l, p in sorted((r for r in rows if r[0] == "table"),
                                             key=lambda r: int(r[1]))]
    assert table == [7, 2, 11]
    for kind, tok, slot in (r for r in rows if r[0] == "slot"):
        assert slot_of(table, int(tok)) == int(slot)


def test_best_of_8_token_counts():
    """'Capítulo 8 ...', section 8.1: 16,800 -> 2,800 with a shared prompt."""
    g = _golden_dict("best_of_8.txt")
    prompt, n, gen = int(g["prompt_tokens"]), int(g["branches"]), int(g["generated_per_branch"])
    # unshared: each branch stores prompt + its own tokens; shared: prompt once
    assert n * (prompt + gen) == int(g["unshared_tokens"])
    assert prompt + n * gen == int(g["shared_tokens"])
    # the same run on the allocator, counted in blocks
    unshared = AllocatorModel(4096)
    for _ in range(n):
        unshared.alloc(blocks_for(prompt + gen))
    assert unshared.stats()[0] == n * 132 == 1056
    shared = AllocatorModel(4096)
    p = shared.alloc(blocks_for(prompt))           # 125 blocks, no partial tail
    for _ in range(n - 1):
        shared.incref(p)
    for _ in range(n):
        shared.alloc(blocks_for(gen))              # 7 private blocks each
    used, free, sh = shared.stats()
    assert used == 125 + n * 7 == 181 and sh == 125


def test_fragmentation_figures():
    for reserved, used, pct, *_ in golden_lines("fragmentation.txt"):
        assert round(100 * internal_waste(int(reserved), int(used))) == int(pct)
    # paged: waste below one block per sequence
    for used in (1, 15, 16, 17, 300, 500, 4095):
        assert blocks_for(used) * 16 - used < 16


def test_branching_saving_tends_to_75_percent():
    """'PagedAttention y Gestión de KV-Cache', section 3.02: up to 75% with 4
    branches -- the shared context stored once instead of 4 times."""
    for L, own in ((2048, 0), (2048, 16), (65536, 16)):
        m = AllocatorModel(100000)
        p = m.alloc(blocks_for(L))
        for _ in range(3):
            m.incref(p)
        for _ in range(4):
            m.alloc(blocks_for(own))
        shared = m.stats()[0]
        unshared = 4 * blocks_for(L + own)
        saving = 1 - shared / unshared
        assert saving <= 0.75 + 1e-12
        if own == 0:
            assert saving == 0.75
    assert saving > 0.749


def test_lifo_order_and_all_or_nothing():
    m = AllocatorModel(8)
    assert m.alloc(3) == [0, 1, 2]
    m.free([1])
    assert m.alloc(2) == [1, 3]
    with pytest.raises(OutOfBlocks):
        m.alloc(5)  # 4 free: nothing taken
    assert m.stats() == (4, 4, 0)
    assert m.alloc(4) == [4, 5, 6, 7]


def test_invalid_requests_change_nothing():
    m = AllocatorModel(4)
    a = m.alloc(2)
    before = (list(m.refcount), list(m.free_stack))
    with pytest.raises(InvalidRequest):
        m.free([a[0], a[0]])        # refcount 1, freed twice
    with pytest.raises(InvalidRequest):
        m.free([3])                 # never allocated
    with pytest.raises(InvalidRequest):
        m.incref([a[0], 2])         # 2 is free
    with pytest.raises(InvalidRequest):
        m.free([7])                 # out of range
    assert (list(m.refcount), list(m.free_stack)) == before


def test_cow_best_of_8_with_partial_tail():
    """2008-token prompt (tail block holds 8 tokens), 8 branches each appending
    64 tokens: branches 0..6 copy the shared tail, branch 7 (last holder)
    writes in place; 126 + 7 + 8*4 = 165 blocks."""
    m = AllocatorModel(1024)
    prompt = m.alloc(blocks_for(2008))
    assert len(prompt) == 126
    tables = []
    for b in range(8):
        if b:
            m.incref(prompt)
        tables.append(list(prompt))
    pairs = []
    for b in range(8):
        pr = m.cow_prepare(tables[b], 2008)
        if pr:
            pairs.append((b, pr))
    assert [b for b, _ in pairs] == list(range(7))
    assert all(src == prompt[-1] for _, (src, _dst) in pairs)
    assert m.refcount[prompt[-1]] == 1
    for b in range(8):
        ctx = 2008
        for _ in range(64):
            if ctx % 16 == 0:
                tables[b] += m.alloc(1)
            ctx += 1
    m.check_invariants(tables)
    assert m.stats()[0] == 165


def test_cow_literal_2000_prompt_has_no_copy():
    m = AllocatorModel(1024)
    prompt = m.alloc(blocks_for(2000))
    tables = [list(prompt)]
    for _ in range(7):
        m.incref(prompt)
        tables.append(list(prompt))
    assert all(m.cow_prepare(t, 2000) is None for t in tables)
    for t in tables:
        for _ in range(4):
            t += m.alloc(1)
    m.check_invariants(tables)
    assert m.stats()[0] == 125 + 8 * 4 == 157
    assert 8 * blocks_for(2064) == 1032  # unshared footprint, for contrast


def test_cancel_returns_every_block():
    """'PagedAttention y Gestión de KV-Cache', section 4.02: freeing a cancelled
    request returns its pages; after all requests end nothing is held."""
    rnd = random.Random(0)
    m = AllocatorModel(256)
    live = []
    for step in range(2000):
        if live and (rnd.random() < 0.45 or m.stats()[1] < 8):
            t = live.pop(rnd.randrange(len(live)))
            m.free(t)
        else:
            t = m.alloc(rnd.randint(1, 6))
            if live and rnd.random() < 0.3:
                src = rnd.choice(live)
                m.incref(src[:2])
                t = src[:2] + t
            live.append(t)
        m.check_invariants(live)
    for t in live:
        m.free(t)
    assert m.stats() == (0, 256, 0)
    assert sorted(m.free_stack) == list(range(256))
