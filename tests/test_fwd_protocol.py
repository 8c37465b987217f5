"""The forward kernels' barrier protocol, simulated on the CPU.

Two schedules, each restated role by role from its kernel and run through
random interleavings (tests/protocol_sim.py checks for deadlocks and for
parity waits that could pass early or alias):

* the one-query-tile kernel (exact_io_aware_tiled_gb300/csrc/fwd_tc1.cu): a
  TMA producer streaming K/V into a ring of NS stages, whose first use of a
  stage skips the empty waits; an S issuer that starts S(s) once the softmax
  has read S(s-1); a P V issuer; the softmax warps;
* the two-query-tile kernels (fwd_tc.cu and fwd_fp8.cu): two slots walking
  the step plan of fwd_plan.cuh, which loads a K/V tile once when both slots
  need it at the same step.  Every loaded stage gets one arrival from each
  slot's P V issuer, after its P V products for a stage it read and once the
  stage has landed for one it did not.  S_x(s) waits for the softmax to have
  read S_x(s-1), or, in fwd_tc.cu at d = 128 where P lies over S, for
  P V_x(s-1).

Planted mistakes must fail: a stage reloaded one step too early, a shared
load released by only one slot, and the early K(0) load from another thread
that once made the producer's first parity wait on a fresh stage hang.
"""
import random

import pytest

from tests.protocol_sim import Bar, Engine, ProtocolError


class OneTile:
    def __init__(self, n, NS, rng, plant=None):
        self.n, self.NS, self.plant = n, NS, plant
        self.engine = Engine(rng)
        self.q_full = Bar("q_full", 1)
        self.s_full, self.s_free = Bar("s_full", 1), Bar("s_free", 1)      # the softmax arrives as one
        self.p_full, self.pv_done = Bar("p_full", 1), Bar("pv_done", 1)
        self.k_full = [Bar("k_full%d" % i, 1) for i in range(NS)]
        self.v_full = [Bar("v_full%d" % i, 1) for i in range(NS)]
        self.k_empty = [Bar("k_empty%d" % i, 1) for i in range(NS)]
        self.v_empty = [Bar("v_empty%d" % i, 1) for i in range(NS)]
        self.nloads = 0

    def load(self, bar):
        self.nloads += 1
        self.engine.later(("tma", self.nloads), bar)

    def early(self):
        # planted: Q and K(0) issued by another thread before the producer runs
        self.load(self.q_full)
        self.load(self.k_full[0])
        return
        yield

    def producer(self):
        NS, n = self.NS, self.n
        if n == 0:
            return
        if self.plant != "early_k0":
            self.load(self.q_full)
        for s in range(n):
            st = s % NS
            first_use = s < (NS + 1 if self.plant == "reload_early" else NS)
            if self.plant == "early_k0" and s == 0:
                yield ("wait", self.k_empty[st], -1)          # the old code's parity-1 wait on a fresh stage
                yield ("wait", self.v_empty[st], -1)
                self.load(self.v_full[st])
                continue
            if not first_use:
                yield ("wait", self.k_empty[st], s // NS - 1)
                yield ("wait", self.v_empty[st], s // NS - 1)
            self.load(self.k_full[st])
            self.load(self.v_full[st])
        for j in range(max(0, n - NS), n):
            yield ("wait", self.k_full[j % NS], j // NS)
            yield ("wait", self.v_full[j % NS], j // NS)
        yield ("wait", self.q_full, 0)

    def s_issuer(self):
        if self.n == 0:
            return
        yield ("wait", self.q_full, 0)
        for s in range(self.n):
            st = s % self.NS
            if s > 0:
                yield ("wait", self.s_free, s - 1)
            yield ("wait", self.k_full[st], s // self.NS)
            self.engine.later("S", self.s_full)
            self.engine.later("S", self.k_empty[st])

    def pv_issuer(self):
        for s in range(self.n):
            st = s % self.NS
            yield ("wait", self.p_full, s)
            yield ("wait", self.v_full[st], s // self.NS)
            self.engine.later("PV", self.pv_done)
            self.engine.later("PV", self.v_empty[st])

    def softmax(self):
        for s in range(self.n):
            yield ("wait", self.s_full, s)
            self.s_free.arrive()
            if s > 0:
                yield ("wait", self.pv_done, s - 1)
            self.p_full.arrive()
        if self.n > 0:
            yield ("wait", self.pv_done, self.n - 1)

    def run(self):
        roles = {"P": self.producer(), "S": self.s_issuer(), "PV": self.pv_issuer(), "SM": self.softmax()}
        if self.plant == "early_k0":
            roles["E"] = self.early()
        self.engine.run(roles)


def step_plan(kvs, s, ld, NS):
    """The loads of step s (stage, absolute phase, kv tile) and the load each
    slot uses: one load when both slots need the same tile, in slot order."""
    loads, use = [], [-1, -1]
    kvA = kvs[0][s] if s < len(kvs[0]) else -1
    kvB = kvs[1][s] if s < len(kvs[1]) else -1
    if kvA >= 0:
        loads.append((ld % NS, ld // NS, kvA))
        ld += 1
        use[0] = 0
    if kvB >= 0:
        if kvB == kvA:
            use[1] = 0
        else:
            loads.append((ld % NS, ld // NS, kvB))
            ld += 1
            use[1] = len(loads) - 1
    return loads, use, ld


class TwoTile:
    def __init__(self, kvs, NS, gate_on_pv, rng, plant=None):
        self.kvs, self.NS, self.gate_on_pv, self.plant = kvs, NS, gate_on_pv, plant
        self.n = [len(kvs[0]), len(kvs[1])]
        self.smax = max(self.n)
        self.engine = Engine(rng)
        self.q_full = Bar("q_full", 1)
        self.s_full = [Bar("s_full%d" % x, 1) for x in range(2)]
        self.s_free = [Bar("s_free%d" % x, 1) for x in range(2)]
        self.p_full = [Bar("p_full%d" % x, 1) for x in range(2)]
        self.pv_done = [Bar("pv_done%d" % x, 1) for x in range(2)]
        self.k_full = [Bar("k_full%d" % i, 1) for i in range(NS)]
        self.v_full = [Bar("v_full%d" % i, 1) for i in range(NS)]
        self.k_empty = [Bar("k_empty%d" % i, 1) for i in range(NS)]
        self.v_empty = [Bar("v_empty%d" % i, 2) for i in range(NS)]     # one arrival per slot
        self.nloads = 0

    def load(self, bar):
        self.nloads += 1
        self.engine.later(("tma", self.nloads), bar)

    def producer(self):
        if self.smax > 0:
            self.load(self.q_full)
        ld = 0
        for s in range(self.smax):
            loads, use, ld = step_plan(self.kvs, s, ld, self.NS)
            for st, ph, _ in loads:
                yield ("wait", self.k_empty[st], ph - 1)
                yield ("wait", self.v_empty[st], ph - 1)
                self.load(self.k_full[st])
                self.load(self.v_full[st])
        for j in range(max(0, ld - self.NS), ld):
            yield ("wait", self.k_full[j % self.NS], j // self.NS)
            yield ("wait", self.v_full[j % self.NS], j // self.NS)
        if self.smax > 0:
            yield ("wait", self.q_full, 0)

    def s_issuer(self):
        if self.smax == 0:
            return
        yield ("wait", self.q_full, 0)
        ld = 0
        for s in range(self.smax):
            loads, use, ld = step_plan(self.kvs, s, ld, self.NS)
            for x in range(2):
                if s >= self.n[x]:
                    continue
                st, ph, _ = loads[use[x]]
                if s > 0:
                    yield ("wait", self.pv_done[x] if self.gate_on_pv else self.s_free[x], s - 1)
                yield ("wait", self.k_full[st], ph)
                self.engine.later("S", self.s_full[x])
            for st, _, _ in loads:
                self.engine.later("S", self.k_empty[st])

    def pv_issuer(self, x):
        if self.smax == 0:
            return
        ld = 0
        for s in range(self.smax):
            loads, use, ld = step_plan(self.kvs, s, ld, self.NS)
            mine = use[x]
            if s < self.n[x]:
                st, ph, _ = loads[mine]
                yield ("wait", self.p_full[x], s)
                yield ("wait", self.v_full[st], ph)
                self.engine.later(("PV", x), self.pv_done[x])
            for l, (st, ph, _) in enumerate(loads):
                if s < self.n[x] and l == mine:
                    self.engine.later(("PV", x), self.v_empty[st])
                elif self.plant != "one_release":
                    yield ("wait", self.v_full[st], ph)
                    self.v_empty[st].arrive()

    def softmax(self, x):
        for s in range(self.n[x]):
            yield ("wait", self.s_full[x], s)
            if not self.gate_on_pv:
                self.s_free[x].arrive()
            if s > 0:
                yield ("wait", self.pv_done[x], s - 1)
            self.p_full[x].arrive()
        if self.n[x] > 0:
            yield ("wait", self.pv_done[x], self.n[x] - 1)

    def run(self):
        self.engine.run({"P": self.producer(), "S": self.s_issuer(), "PV0": self.pv_issuer(0),
                         "PV1": self.pv_issuer(1), "SM0": self.softmax(0), "SM1": self.softmax(1)})


def _slot_pairs(rng):
    """kv tile lists of two slots in the shapes the masks give: causal rows of
    two query tiles, dense rows, sliding windows, block-sparse lists, and
    slots with nothing to do."""
    kind = rng.randrange(5)
    if kind == 0:                                   # causal: tiles 0..qt
        qa = rng.randrange(0, 9)
        qb = qa + rng.randrange(0, 3)
        return [list(range(qa + 1)), list(range(qb + 1))]
    if kind == 1:                                   # dense (key padding: fewer tiles)
        m = rng.randrange(1, 9)
        return [list(range(m)), list(range(m))]
    if kind == 2:                                   # sliding window
        la, lb = rng.randrange(0, 4), rng.randrange(0, 4)
        return [list(range(la, la + rng.randrange(1, 5))), list(range(lb, lb + rng.randrange(1, 5)))]
    if kind == 3:                                   # block-sparse
        return [sorted(rng.sample(range(12), rng.randrange(1, 7))), sorted(rng.sample(range(12), rng.randrange(1, 7)))]
    one = list(range(rng.randrange(1, 6)))          # one slot past the last query tile
    return [one, []] if rng.random() < 0.5 else [[], one]


@pytest.mark.parametrize("NS", [2, 3, 5])
def test_one_tile_forward_protocol(NS):
    rng = random.Random(31 + NS)
    for n in list(range(0, 9)) + [rng.randrange(9, 40) for _ in range(10)]:
        for _ in range(15):
            OneTile(n, NS, random.Random(rng.random())).run()


@pytest.mark.parametrize("NS,gate_on_pv", [(5, False), (2, True), (3, False), (2, False)])
def test_two_tile_forward_protocol(NS, gate_on_pv):
    rng = random.Random(71 + NS + 10 * gate_on_pv)
    for _ in range(400):
        TwoTile(_slot_pairs(rng), NS, gate_on_pv, random.Random(rng.random())).run()
    TwoTile([[], []], NS, gate_on_pv, random.Random(0)).run()


@pytest.mark.parametrize("plant", ["reload_early", "early_k0"])
def test_one_tile_planted_mistakes_are_caught(plant):
    rng = random.Random(5)
    with pytest.raises(ProtocolError):
        for _ in range(300):
            OneTile(rng.randrange(4, 12), 3, random.Random(rng.random()), plant=plant).run()


def test_two_tile_planted_mistake_is_caught():
    rng = random.Random(6)
    with pytest.raises(ProtocolError):
        for _ in range(300):
            TwoTile(_slot_pairs(rng), 5, False, random.Random(rng.random()), plant="one_release").run()
