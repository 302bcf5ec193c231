"""A small discrete-event simulator for host models of the kernels' barrier protocols (test
infrastructure).  Actors are generators that yield ("until", predicate) to block until the
predicate holds, or ("sleep", dt) to take time; timed callbacks (a copy landing, a product
completing) run from the same event queue.  Blocked actors wake a random short time after
their predicate becomes true, as a waiting warp sees a barrier phase complete."""
import heapq


class Sim:
    """Actors are generators that yield ("until", predicate) or ("sleep", dt); timed
    callbacks (a load landing, a product completing) run from the same event queue."""

    def __init__(self, rng):
        self.rng, self.now, self.seq, self.q = rng, 0.0, 0, []
        self.blocked = []  # (predicate, actor)

    def at(self, t, fn):
        self.seq += 1
        heapq.heappush(self.q, (t, self.seq, fn))

    def start(self, actor):
        self.at(self.now, lambda: self.step(actor))

    def step(self, actor):
        try:
            kind, arg = next(actor)
        except StopIteration:
            return
        if kind == "sleep":
            self.at(self.now + arg, lambda: self.step(actor))
        elif arg():
            self.at(self.now + self.rng.uniform(0.0, 0.05), lambda: self.step(actor))
        else:
            self.blocked.append((arg, actor))

    def run(self, limit=500000):
        for _ in range(limit):
            if not self.q:
                return
            self.now, _, fn = heapq.heappop(self.q)
            fn()
            ready = [(p, a) for p, a in self.blocked if p()]
            self.blocked = [(p, a) for p, a in self.blocked if not p()]
            for _, a in ready:  # wake-up latency
                self.at(self.now + self.rng.uniform(0.0, 0.05), lambda a=a: self.step(a))
        raise AssertionError("the model did not finish")
