"""A model check, on the CPU, of the mbarrier protocol of the tcgen05 prefill
kernel (one CTA, one query tile of n 128-key blocks).

Every role of the kernel (the TMA producer, the MMA-issuing thread, the four
V-converter warps, the eight softmax warps) is an agent that issues, in the
kernel's order, the same waits and arrivals on the same barriers; the tensor
pipe runs the issued MMAs in order and a commit arrives once every MMA before
it is done.  Delays are random, and so is the time a waiting thread takes to
notice that its phase completed (the kernel's waits sleep, and a sleeping
thread may wake late).

An mbarrier wait names a phase only by its parity, so it is correct only if,
when the wait starts, the barrier has completed either all phases before the
awaited one or the awaited one too, and if the barrier does not complete the
phase after it before the waiter has returned.  The check asserts both for
every wait, and that every run ends (no deadlock).  The kernel's protocol
passes on thousands of random schedules; the earlier protocol with a single
barrier for every block's P (which a schedule with a late-waking MMA thread
breaks, as it did on the GPU) is found to fail, which shows the model can
tell."""
import random

import pytest

from barrier_model import Agent, Sim, Violation


def prefill_cta(rng, n, fp8, single_p, rescale_p=0.02, blk=False):
    """The barriers and roles of one CTA of the tcgen05 prefill over n blocks
    (blk: a block-scaled FP8 pool, whose page scales go to the softmax warps
    through a two-buffer hand-off of their own)."""
    R = 2 if fp8 else 3
    d = lambda lo, hi: ("delay", rng.uniform(lo, hi))

    def bars(sim):
        for i in range(R):
            sim.bar(f"kv_full{i}", 1)
            sim.bar(f"kv_empty{i}", 5 if fp8 else 1)
        for i in range(2):
            sim.bar(f"s_full{i}", 1)
            sim.bar(f"vt_full{i}", 4)
            sim.bar(f"vt_empty{i}", 1)
            sim.bar(f"p_full{i}", 8)
            sim.bar(f"sc_full{i}", 1)
            sim.bar(f"sc_empty{i}", 8)
        sim.bar("p_full", 8)
        for name, c in (("q_ready", 8), ("drain", 1), ("xchg", 8), ("tail_ready", 1), ("tail_done", 4)):
            sim.bar(name, c)

    def p_bar(j):  # the barrier P(j) is signalled on, and the phase it completes
        return ("p_full", j) if single_p else (f"p_full{j % 2}", j // 2)

    def producer():
        for j in range(n):
            if j >= R:
                yield ("wait", f"kv_empty{j % R}", j // R - 1)
            if blk:  # the block's page scales into buffer j % 2
                if j >= 2:
                    yield ("wait", f"sc_empty{j % 2}", j // 2 - 1)
                yield ("arrive", [f"sc_full{j % 2}"])
            yield d(0.0, 0.3)
            yield ("tma", f"kv_full{j % R}")
        for x in range(max(0, n - R), n):  # no copy in flight at the end
            yield ("wait", f"kv_full{x % R}", x // R)

    def mma():
        yield ("wait", "q_ready", 0)

        def qk(j):
            yield ("wait", f"kv_full{j % R}", j // R)
            if not fp8 and j == n - 1:
                yield ("arrive", ["tail_ready"])
            yield d(0.0, 0.4)  # issuing takes the thread a while
            yield ("mma", [f"s_full{j % 2}"] + ([f"kv_empty{j % R}"] if fp8 else []))

        for j in range(min(2, n)):
            yield from qk(j)
        for i in range(n):
            yield ("wait",) + p_bar(i)
            if fp8:
                yield ("wait", f"vt_full{i % 2}", i // 2)
            elif i == n - 1:
                yield ("wait", "tail_done", 0)
            yield d(0.0, 0.4)
            yield ("mma", [f"vt_empty{i % 2}"] if fp8 else [f"kv_empty{i % R}"])
            if i + 2 < n:
                yield from qk(i + 2)
        yield ("mma", ["drain"])
        yield ("wait", "drain", 0)

    def converter():
        if fp8:
            for j in range(n):
                yield ("wait", f"kv_full{j % R}", j // R)
                if j >= 2:
                    yield ("wait", f"vt_empty{j % 2}", j // 2 - 1)
                yield d(0.2, 1.0)
                yield ("arrive", [f"vt_full{j % 2}", f"kv_empty{j % R}"])
        else:
            yield ("wait", "tail_ready", 0)
            yield ("wait", f"kv_full{(n - 1) % R}", (n - 1) // R)
            yield d(0.0, 0.3)
            yield ("arrive", ["tail_done"])

    def softmax():
        xk = 0

        def exchange():
            nonlocal xk
            yield ("arrive", ["xchg"])
            yield ("wait", "xchg", xk)
            xk += 1

        yield d(0.2, 2.0)  # Q into TMEM
        yield from exchange()
        yield ("arrive", ["q_ready"])
        for j in range(n):
            if blk:
                yield ("wait", f"sc_full{j % 2}", j // 2)
            yield ("wait", f"s_full{j % 2}", j // 2)
            yield d(0.1, 0.8)
            yield from exchange()
            if j > 0 and rng.random() < rescale_p:  # O rescaled after P V(j - 1) (rare: the max grew by 2^8)
                if fp8:
                    yield ("wait", f"vt_empty{(j - 1) % 2}", (j - 1) // 2)
                else:
                    yield ("wait", f"kv_empty{(j - 1) % R}", (j - 1) // R)
            yield d(0.3, 1.5)
            name, _ = p_bar(j)
            yield ("arrive", ([f"sc_empty{j % 2}"] if blk else []) + [name])
        yield from exchange()
        yield ("wait", "drain", 0)

    agents = [Agent("producer", producer()), Agent("mma", mma())]
    agents += [Agent(f"conv{i}", converter()) for i in range(4)]
    agents += [Agent(f"softmax{i}", softmax()) for i in range(8)]
    return bars, agents


def run_once(seed, n, fp8, single_p, wake_max, blk=False):
    rng = random.Random(seed)
    sim = Sim(rng, wake_max)
    bars, agents = prefill_cta(rng, n, fp8, single_p, blk=blk)
    bars(sim)
    sim.run(agents)


@pytest.mark.parametrize("fp8,blk", [(True, False), (True, True), (False, False)])
def test_kernel_protocol_holds_on_random_schedules(fp8, blk):
    for seed in range(600):
        for n in (1, 2, 3, 4, 5, 8):
            run_once(seed * 31 + n, n, fp8, single_p=False, wake_max=25.0, blk=blk)


@pytest.mark.parametrize("fp8", [True, False])
def test_single_p_barrier_is_caught(fp8):
    """The protocol before the fix: one barrier for every block's P.  A
    late-waking MMA thread lets the softmax complete P(j) and P(j + 1) first."""
    found = 0
    for seed in range(300):
        try:
            run_once(seed, 6, fp8, single_p=True, wake_max=25.0)
        except Violation as e:
            assert "p_full" in str(e), str(e)
            found += 1
    assert found > 0, "the model did not find the single-barrier hazard"
