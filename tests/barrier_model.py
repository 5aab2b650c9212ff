"""An event-driven model of CTA roles synchronising through mbarriers, for
checking a kernel's barrier protocol on the CPU (tests/test_*_barrier_model.py).

An agent is a generator of actions: ("wait", barrier, phase), ("arrive",
[barriers]), ("delay", t), ("tma", barrier) (one arrival when the copy
lands), ("mma", [barriers]) (one arrival each once this and every earlier
MMA are done).  Delays are random, and so is the time a waiting agent takes
to notice that its phase completed: mostly at once, now and then late.

An mbarrier wait names a phase only by its parity, so it is correct only if,
when it starts, the barrier has completed either all phases before the
awaited one or the awaited one too, and if the barrier does not complete the
phase after it before the waiter has returned.  Sim raises Violation when
either fails, and when a run ends with agents still waiting (deadlock)."""
import heapq


class Violation(Exception):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, 0, 0
        self.waiters = []  # [agent, phase, released]


class Sim:
    def __init__(self, rng, wake_max):
        self.rng, self.wake_max = rng, wake_max
        self.t, self.seq, self.q = 0.0, 0, []
        self.bars = {}
        self.agents_live = 0
        self.pipe_free = 0.0  # the tensor pipe runs issued MMAs in order

    def bar(self, name, count):
        self.bars[name] = Barrier(name, count)

    def wake_delay(self):
        # most waiters notice at once; now and then one sleeps on (up to the
        # kernel's 20 us suspend hint)
        return self.rng.uniform(0, 0.2) if self.rng.random() < 0.9 else self.rng.uniform(0, self.wake_max)

    def at(self, dt, fn):
        self.seq += 1
        heapq.heappush(self.q, (self.t + dt, self.seq, fn))

    def arrive(self, name):
        b = self.bars[name]
        b.pending += 1
        if b.pending == b.count:
            b.pending = 0
            b.done += 1
            for w in b.waiters:
                agent, phase, released = w
                if b.done > phase + 1:
                    raise Violation(f"{b.name} completed phase {b.done - 1} while {agent.name} "
                                    f"still waited for phase {phase}")
                if not released and b.done == phase + 1:
                    w[2] = True
                    self.at(self.wake_delay(), lambda a=agent, ww=w, bb=b: self.wake(a, bb, ww))

    def wake(self, agent, b, w):
        b.waiters.remove(w)
        self.step(agent)

    def wait(self, agent, name, phase):
        b = self.bars[name]
        if not (phase <= b.done <= phase + 1):
            raise Violation(f"{agent.name} waits for phase {phase} of {name}, which has completed "
                            f"{b.done}")
        w = [agent, phase, b.done == phase + 1]
        b.waiters.append(w)
        if w[2]:
            self.at(self.wake_delay(), lambda: self.wake(agent, b, w))

    def mma(self, commits):
        """Issue one MMA group; each named barrier gets one arrival once it
        and every MMA before it are done."""
        start = max(self.t, self.pipe_free)
        self.pipe_free = start + self.rng.uniform(0.05, 0.6)
        for c in commits:
            self.at(self.pipe_free - self.t, lambda c=c: self.arrive(c))

    def step(self, agent):
        try:
            op = next(agent.gen)
        except StopIteration:
            self.agents_live -= 1
            return
        kind = op[0]
        if kind == "wait":
            self.wait(agent, op[1], op[2])
        elif kind == "delay":
            self.at(op[1], lambda: self.step(agent))
        elif kind == "arrive":
            for name in op[1]:
                self.arrive(name)
            self.at(0, lambda: self.step(agent))
        elif kind == "tma":  # the copy lands later; the issuer goes on
            self.at(self.rng.uniform(0.1, 4.0), lambda n=op[1]: self.arrive(n))
            self.at(0, lambda: self.step(agent))
        elif kind == "mma":
            self.mma(op[1])
            self.at(0, lambda: self.step(agent))

    def run(self, agents):
        self.agents_live = len(agents)
        for a in agents:
            self.at(0, lambda a=a: self.step(a))
        while self.q:
            self.t, _, fn = heapq.heappop(self.q)
            fn()
        if self.agents_live:
            stuck = [f"{b.name}:{w[0].name}@{w[1]}" for b in self.bars.values() for w in b.waiters]
            raise Violation(f"deadlock: {stuck}")


class Agent:
    def __init__(self, name, gen):
        self.name, self.gen = name, gen
