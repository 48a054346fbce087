"""Discrete-event core for the barrier-protocol models in test_*_protocol.py (test code only).

Agents are generators that yield ("delay", dt), ("wait", predicate) or ("twait", predicate,
limit); a bounded wait resumes the agent with True once the predicate holds, or with False
when `limit` time passes first (the kernels' time-limited mbarrier waits).  Barriers model
mbarrier phases (arrival count plus transaction count) and check every parity wait for
ambiguity; the tensor pipe runs one issuing thread's MMAs in order and lands a commit's
arrival when every earlier MMA has finished.
"""
import heapq
import itertools


class Hazard(AssertionError):
    pass


class Bar:
    """An mbarrier: `count` arrivals plus a transaction count complete a phase."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.done = name, count, count, 0, 0

    def arrive(self, expect=0):
        self.tx += expect
        self.pending -= 1
        if self.pending < 0:
            raise Hazard(f"{self.name}: more arrivals than its count in one phase")
        self._check()

    def expect(self, nbytes):
        self.tx += nbytes

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count

    def passed(self, phase, hw=False):
        """Parity wait for `phase`: true once it completed; ambiguous states are errors.

        hw=True answers as the hardware's parity test does (the current phase's parity
        differs from the awaited one's) without the ambiguity check, for waits whose
        consequences the caller checks otherwise."""
        if hw:
            return self.done % 2 != phase % 2
        if self.done not in (phase, phase + 1):
            raise Hazard(f"{self.name}: waiting for phase {phase} with {self.done} completed")
        return self.done == phase + 1


class Sim:
    def __init__(self, rng):
        self.rng, self.t, self.events, self.waiters = rng, 0.0, [], []
        self.seq = itertools.count()
        self.finished = set()
        self.finish_time = {}

    def at(self, dt, fn):
        heapq.heappush(self.events, (self.t + dt, next(self.seq), fn))

    def start(self, name, gen):
        self._step(name, gen)

    def _step(self, name, gen, value=None):
        while True:
            try:
                req = gen.send(value)
            except StopIteration:
                self.finished.add(name)
                self.finish_time[name] = self.t
                return
            if req[0] == "delay":
                self.at(req[1], lambda: self._step(name, gen, None))
                return
            if req[1]():  # "wait" or "twait": already true
                value = True
                continue
            w = (name, gen, req[1])
            self.waiters.append(w)
            if req[0] == "twait":
                def expire(w=w):
                    if w in self.waiters:
                        self.waiters.remove(w)
                        self._step(w[0], w[1], False)
                self.at(req[2], expire)
            return

    def _poll(self):
        progress = True
        while progress:
            progress = False
            for w in list(self.waiters):
                if w in self.waiters and w[2]():
                    self.waiters.remove(w)
                    self._step(w[0], w[1], True)
                    progress = True

    def run(self):
        self._poll()
        while self.events:
            self.t, _, fn = heapq.heappop(self.events)
            fn()
            self._poll()
        if self.waiters:
            raise Hazard("deadlock: " + ", ".join(w[0] for w in self.waiters))


class TensorPipe:
    """One issuing thread's MMAs run in issue order; a commit arrives when all earlier finish."""

    def __init__(self, sim):
        self.sim, self.free_at = sim, 0.0

    def mma(self, dur, on_start, on_end):
        start = max(self.sim.t, self.free_at)
        self.free_at = start + dur
        self.sim.at(start - self.sim.t, on_start)
        self.sim.at(self.free_at - self.sim.t, on_end)

    def commit(self, bar):
        self.sim.at(max(0.0, self.free_at - self.sim.t), bar.arrive)
