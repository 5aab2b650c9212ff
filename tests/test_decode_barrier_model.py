"""A model check, on the CPU, of the mbarrier protocols of the decode kernels
(barrier_model.py says what is checked).

decode_kernel (fixed splits): a producer lane streams the split's pages into
an 8-stage ring (full[s] completes when a page's two copies land, empty[s]
when its consumer warp is done with it); consumer warp w takes pages
w, w + 4, ...

decode_bal_kernel (balanced schedule): the CTA's range crosses units (one
sequence and KV head each).  Ahead of each unit the producer stages its query
rows and descriptor (q_full: one copy), once the four consumer warps have
taken the previous unit's (q_empty: one arrival each); the pages of all its
units share one ring, and consumer warp w takes the CTA's pages w, w + 4, ...
whatever unit they belong to.

Both pass on random schedules; a producer that staged a unit's query rows
without waiting for q_empty is caught."""
import random

import pytest

from barrier_model import Agent, Sim, Violation

STAGES, WARPS = 8, 4


def decode_cta(rng, unit_pages, balanced, skip_q_empty=False):
    d = lambda lo, hi: ("delay", rng.uniform(lo, hi))
    n = sum(unit_pages)

    def bars(sim):
        for s in range(STAGES):
            sim.bar(f"full{s}", 1)
            sim.bar(f"empty{s}", 1)
        sim.bar("q_full", 1)
        sim.bar("q_empty", WARPS)

    def producer():
        k = 0
        for j, len_j in enumerate(unit_pages if balanced else [n]):
            if balanced:
                if j > 0 and not skip_q_empty:
                    yield ("wait", "q_empty", j - 1)
                yield ("tma", "q_full")
            for _ in range(len_j):
                if k >= STAGES:
                    yield ("wait", f"empty{k % STAGES}", k // STAGES - 1)
                yield d(0.0, 0.2)
                yield ("tma", f"full{k % STAGES}")
                k += 1
        # no copy in flight at the end: each stage's last use, and the last query rows
        for s in range(min(STAGES, k)):
            uses = (k - 1 - s) // STAGES + 1
            yield ("wait", f"full{s}", uses - 1)
        if balanced and unit_pages:
            yield ("wait", "q_full", len(unit_pages) - 1)

    def consumer(w):
        kb = 0
        for j, len_j in enumerate(unit_pages if balanced else [n]):
            if balanced:
                yield ("wait", "q_full", j)
                yield d(0.0, 0.5)  # query rows into registers
                yield ("arrive", ["q_empty"])
            for k in range(kb + ((w - kb) % WARPS), kb + len_j, WARPS):
                yield ("wait", f"full{k % STAGES}", k // STAGES)
                yield d(0.2, 1.0)
                yield ("arrive", [f"empty{k % STAGES}"])
            kb += len_j
            yield d(0.0, 0.5)  # the four warps' merge (a named barrier: no phases)

    agents = [Agent("producer", producer())] + [Agent(f"consumer{w}", consumer(w)) for w in range(WARPS)]
    return bars, agents


def run_once(seed, balanced, skip_q_empty=False):
    rng = random.Random(seed)
    units = [rng.choice([1, 2, 3, 5, 9, 17, 40]) for _ in range(rng.randint(1, 6))]
    sim = Sim(rng, 25.0)
    bars, agents = decode_cta(rng, units, balanced, skip_q_empty)
    bars(sim)
    sim.run(agents)


@pytest.mark.parametrize("balanced", [False, True])
def test_decode_protocols_hold_on_random_schedules(balanced):
    for seed in range(1500):
        run_once(seed, balanced)


def test_query_staging_without_its_wait_is_caught():
    found = 0
    for seed in range(300):
        try:
            run_once(seed, True, skip_q_empty=True)
        except Violation as e:
            assert "q_full" in str(e) or "q_empty" in str(e), str(e)
            found += 1
    assert found > 0, "the model did not find the missing q_empty wait"
