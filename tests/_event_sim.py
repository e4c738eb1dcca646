"""A small discrete-event engine for checking a kernel's mbarrier protocol
on the CPU: roles are generators that yield ("wait", barrier, parity,
intended completed phases, site) or ("delay", dt); a barrier completes a
phase when its arrivals and transaction bytes are all in, and a parity
test passes as on the device (the last completed phase has the other
parity).  A wait that passes on a phase count other than the intended one
(two phases ahead, say) is reported, as is a role that never finishes."""

import heapq
import random


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.completed = name, count, count, 0, 0

    def test(self, parity):
        return (self.completed & 1) != parity


class EventSim:
    def __init__(self, seed):
        self.rng = random.Random(seed)
        self.now = 0.0
        self.events = []
        self.seq = 0
        self.waiting = []  # (bar, parity, gen, intended, site)
        self.violations = []
        self.done = set()

    def at(self, t, fn):
        self.seq += 1
        heapq.heappush(self.events, (t, self.seq, fn))

    def fail(self, msg):
        self.violations.append(f"t={self.now:.2f}: {msg}")

    def arrive(self, bar, n=1):
        bar.pending -= n
        self._maybe_complete(bar)

    def expect_tx(self, bar, nbytes):
        bar.tx += nbytes
        self.arrive(bar)

    def complete_tx(self, bar, nbytes):
        bar.tx -= nbytes
        self._maybe_complete(bar)

    def copy(self, bar, nbytes, land, lo=0.5, hi=6.0):
        """An asynchronous copy: `land` runs when its bytes arrive."""

        def fin():
            land()
            self.complete_tx(bar, nbytes)

        self.at(self.now + self.rng.uniform(lo, hi), fin)

    def _maybe_complete(self, bar):
        if bar.pending == 0 and bar.tx == 0:
            bar.completed += 1
            bar.pending = bar.count
            still = []
            for w in self.waiting:
                if w[0] is bar and bar.test(w[1]):
                    self.at(self.now, lambda w=w: self._resume(w))
                else:
                    still.append(w)
            self.waiting = still

    def _check(self, bar, intended, site):
        if bar.completed != intended:
            self.fail(f"{site}: {bar.name} has completed {bar.completed} phases, wanted {intended}")

    def _resume(self, w):
        bar, _, gen, intended, site = w
        self._check(bar, intended, site)
        self.step(gen)

    def step(self, gen):
        try:
            req = next(gen)
        except StopIteration:
            return
        if req[0] == "delay":
            self.at(self.now + req[1], lambda: self.step(gen))
        else:
            _, bar, parity, intended, site = req
            if bar.test(parity):
                self._check(bar, intended, site)
                self.at(self.now, lambda: self.step(gen))
            else:
                self.waiting.append((bar, parity, gen, intended, site))

    def run_roles(self, roles, expect_done):
        for g in roles:
            self.at(0.0, lambda g=g: self.step(g))
        while self.events:
            self.now, _, fn = heapq.heappop(self.events)
            fn()
        if self.done != set(expect_done):
            self.fail(f"deadlock: finished {sorted(self.done)}, waiting on {sorted(w[0].name for w in self.waiting)}")
        return self.violations
