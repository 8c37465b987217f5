"""A small simulator of mbarrier protocols, for the kernels' CPU tests.

A kernel role is a Python generator that yields ("wait", bar, k) to block
until phase k of `bar` is complete (k = -1: the phase before the first,
complete from the start), calls `Bar.arrive()` for a plain arrival, and
queues asynchronous arrivals (a tcgen05 commit, a TMA load's completion) on a
FIFO of its own through `Engine.later(fifo, bar)`: each FIFO fires in order,
at a time the scheduler picks.  `Engine.run` interleaves the roles and the
FIFOs at random and raises ProtocolError on

* a deadlock (no role can move and nothing is in flight);
* a wait that the hardware's parity test would pass at once although phase
  k is not complete (phase k - 1 still open when the wait starts);
* a waiter whose barrier has run two or more phases past the phase it waits
  for (the parity would alias).
"""


class ProtocolError(AssertionError):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.completed = name, count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.completed += 1


class Engine:
    def __init__(self, rng):
        self.rng = rng
        self.fifos = {}

    def later(self, fifo, bar):
        self.fifos.setdefault(fifo, []).append(bar)

    def run(self, roles, max_events=10 ** 6):
        roles = dict(roles)
        waiting = {}

        def advance(name):
            try:
                _, bar, k = next(roles[name])
            except StopIteration:
                del roles[name]
                waiting.pop(name, None)
                return
            if bar.completed < k:
                raise ProtocolError("%s starts waiting for phase %d of %s while phase %d is incomplete: "
                                    "the parity wait would pass at once" % (name, k, bar.name, k - 1))
            waiting[name] = (bar, k)

        for name in list(roles):
            advance(name)
        for _ in range(max_events):
            for name, (bar, k) in waiting.items():
                if bar.completed > k + 1:
                    raise ProtocolError("%s waits for phase %d of %s, which is already %d phases on: "
                                        "the parity aliases" % (name, k, bar.name, bar.completed - k))
            ready = [n for n, (bar, k) in waiting.items() if bar.completed >= k + 1]
            fifos = [f for f, q in self.fifos.items() if q]
            choices = [("role", n) for n in ready] + [("async", f) for f in fifos]
            if not choices:
                if roles:
                    raise ProtocolError("deadlock: %s" % ", ".join(
                        "%s waits %s phase %d (completed %d)" % (n, b.name, k, b.completed)
                        for n, (b, k) in waiting.items()))
                return
            kind, x = choices[self.rng.randrange(len(choices))]
            if kind == "role":
                advance(x)
            else:
                self.fifos[x].pop(0).arrive()
        raise ProtocolError("no end after %d events" % max_events)
