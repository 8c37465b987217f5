"""The backward kernels' barrier protocol, simulated on the CPU.

The persistent backward kernels (exact_io_aware_tiled_gb300/csrc/bwd_tc.cu
at head dimension 64, bwd_tc128.cu at 128) run five roles that meet only at mbarriers: the TMA producer (which also
claims work items and issues the dQ reduce-adds), the S^T / dP^T issuer, the
dV / dK issuer, the dQ issuer and the compute warps.  This test restates each
role's sequence of waits and arrivals as those files issue them (phases by
their absolute index, asynchronous completions -- TMA loads and tcgen05
commits -- as events that fire at some later time) and runs random
interleavings over random work-item sequences, with and without the
dropout variant's item-claim order.  At d = 64, K is double-buffered per item
and V has a buffer of its own; at d = 128 K and V share one load and one
buffer, and each 128-row query tile is two 64-row steps.  It checks that

* every run finishes (no interleaving deadlocks);
* no parity wait could pass early: when a role starts waiting for phase k,
  phase k - 1 is complete (were it still open, the parity test would read
  phase k as complete at once);
* no barrier runs two phases past a waiter that has not yet seen phase k
  (the parity would then alias);
* the producer's four-entry ring of step coordinates still holds step r
  when the reduce of step r reads it.

A mistake planted in the simulated protocol (the reduce issued before its
staging buffer is full, or a fourth load issued into a three-stage ring)
must make it fail.
"""
import random

import pytest

from tests.protocol_sim import Bar, Engine, ProtocolError

NSB = 3      # Q / dO ring stages
NSTG = 1     # float32 dQ staging buffers
KLAG = 3     # the dQ reduce of step g - KLAG follows the loads of step g


class Sim:
    """The five roles of one CTA as generators (tests/protocol_sim.py)."""

    def __init__(self, items, drop, rng, plant=None, d=64):
        self.items, self.drop, self.rng, self.plant, self.d = items, drop, rng, plant, d
        self.per_tile = 1 if d == 64 else 2                               # steps per query tile
        B = Bar
        self.item_full = [B("item_full%d" % i, 1) for i in range(2)]
        self.item_empty = [B("item_empty%d" % i, 4) for i in range(2)]   # three issuers + the compute warps
        self.k_full = [B("k_full%d" % i, 1) for i in range(2)]
        self.k_empty = [B("k_empty%d" % i, 2) for i in range(2)]          # S^T issuer and dQ issuer
        self.q_full = [B("q_full%d" % i, 1) for i in range(NSB)]
        self.q_empty = [B("q_empty%d" % i, 1) for i in range(NSB)]
        self.v_full, self.v_empty = B("v_full", 1), B("v_empty", 1)      # d = 64
        self.kv_full, self.kv_empty = B("kv_full", 1), B("kv_empty", 2)   # d = 128: S^T / dP^T and dQ issuers
        for n in ("s_full", "p_full", "dp_full", "ds_full", "dq_full", "dq_free", "dkv_full", "pt_free"):
            setattr(self, n, B(n, 1))
        self.dsm_free = B("dsm_free", 2)                                  # dK and dQ read the dS^T tile
        self.stg_full = [B("stg_full%d" % i, 1) for i in range(NSTG)]
        self.stg_free = [B("stg_free%d" % i, 1) for i in range(NSTG)]
        self.mailbox = [None, None]
        self.info = [None] * 4
        self.engine = Engine(rng)
        self.nloads = 0

    # asynchronous arrivals: tcgen05 commits complete in issue order per
    # thread; TMA loads in any order
    def commit(self, who, bar):
        self.engine.later(who, bar)

    def load(self, bar):
        self.nloads += 1
        self.engine.later(("tma", self.nloads), bar)

    # ------------------------------------------------------------------ roles
    def producer(self):
        st = {"g": 0, "nkv": 0, "rd": 0, "kf": 0, "next": 0, "loaded": -1}

        def reduce(r):
            if self.plant != "reduce_unstaged":
                yield ("wait", self.stg_full[r % NSTG], r // NSTG)
            if self.stg_full[r % NSTG].completed < r // NSTG + 1:
                raise ProtocolError("reduce of step %d before its dQ was staged" % r)
            if st["loaded"] - r >= 4 or self.info[r & 3] != r:
                raise ProtocolError("step coordinates of %d overwritten before its reduce" % r)
            self.stg_free[r % NSTG].arrive()        # after cp.async.bulk.wait_group.read 0

        def reduce_to(last):
            while st["rd"] <= last:
                yield from reduce(st["rd"])
                st["rd"] += 1

        def publish():
            slot = st["kf"] & 1
            yield ("wait", self.item_empty[slot], (st["kf"] >> 1) - 1)
            v = st["next"] if st["next"] < len(self.items) else -1
            st["next"] += 1
            self.mailbox[slot] = v
            self.item_full[slot].arrive()
            st["kf"] += 1
            return v

        while True:
            if not self.drop:
                yield from reduce_to(st["g"] - KLAG)
            u = yield from publish()
            if u < 0:
                break
            steps = self.items[u] * self.per_tile
            if steps == 0:
                yield from reduce_to(st["g"] - 3)
                continue
            if self.d == 64:
                kb = st["nkv"] & 1
                yield ("wait", self.k_empty[kb], (st["nkv"] >> 1) - 1)
                self.load(self.k_full[kb])
            else:
                yield ("wait", self.kv_empty, st["nkv"] - 1)
                self.load(self.kv_full)
            vi = st["nkv"]
            st["nkv"] += 1
            for t in range(steps):
                g = st["g"]
                nsb = NSB + 1 if self.plant == "ring_too_deep" else NSB
                if self.plant == "ring_too_deep":
                    yield ("wait", self.q_empty[g % NSB], g // nsb - 1)
                else:
                    yield ("wait", self.q_empty[g % NSB], g // NSB - 1)
                self.load(self.q_full[g % NSB])
                self.info[g & 3] = g
                st["loaded"] = g
                if t == 0 and self.d == 64:
                    yield ("wait", self.v_empty, vi - 1)
                    self.load(self.v_full)
                yield from reduce_to(g - KLAG)
                st["g"] += 1
        yield from reduce_to(st["g"] - 1)

    def fetch(self, who, kc):
        slot = kc & 1
        yield ("wait", self.item_full[slot], kc >> 1)
        v = self.mailbox[slot]
        self.item_empty[slot].arrive()
        return v

    def s_issuer(self):
        g = nkv = kc = 0
        while True:
            u = yield from self.fetch("S", kc)
            kc += 1
            if u < 0:
                break
            steps = self.items[u] * self.per_tile
            if steps == 0:
                continue
            kb = nkv & 1
            if self.d == 64:
                yield ("wait", self.k_full[kb], nkv >> 1)
            else:
                yield ("wait", self.kv_full, nkv)
            vi = nkv
            nkv += 1
            for t in range(steps):
                if g > 0:
                    yield ("wait", self.p_full, g - 1)
                yield ("wait", self.q_full[g % NSB], g // NSB)
                self.commit("S", self.s_full)
                if g > 0:
                    yield ("wait", self.ds_full, g - 1)
                if t == 0 and self.d == 64:
                    yield ("wait", self.v_full, vi)
                self.commit("S", self.dp_full)
                g += 1
            if self.d == 64:
                self.commit("S", self.k_empty[kb])
                self.commit("S", self.v_empty)
            else:
                self.commit("S", self.kv_empty)

    def dvdk_issuer(self):
        g = kc = 0
        while True:
            u = yield from self.fetch("D", kc)
            kc += 1
            if u < 0:
                break
            steps = self.items[u] * self.per_tile
            if steps == 0:
                continue
            for t in range(steps):
                yield ("wait", self.p_full, g)
                yield ("wait", self.q_full[g % NSB], g // NSB)
                self.commit("D", self.pt_free)
                yield ("wait", self.ds_full, g)
                self.commit("D", self.dsm_free)
                self.commit("D", self.q_empty[g % NSB])
                g += 1
            self.commit("D", self.dkv_full)

    def dq_issuer(self):
        g = nkv = kc = 0
        while True:
            u = yield from self.fetch("Q", kc)
            kc += 1
            if u < 0:
                break
            steps = self.items[u] * self.per_tile
            if steps == 0:
                continue
            kb = nkv & 1
            nkv += 1
            for t in range(steps):
                yield ("wait", self.ds_full, g)
                if g > 0:
                    yield ("wait", self.dq_free, g - 1)
                self.commit("Q", self.dq_full)
                self.commit("Q", self.dsm_free)
                g += 1
            self.commit("Q", self.k_empty[kb] if self.d == 64 else self.kv_empty)

    def compute(self):
        t = nit = kc = 0

        def drain(r):
            yield ("wait", self.dq_full, r)
            self.dq_free.arrive()
            if r >= NSTG:
                yield ("wait", self.stg_free[r % NSTG], (r - NSTG) // NSTG)
            self.stg_full[r % NSTG].arrive()

        while True:
            u = yield from self.fetch("C", kc)
            kc += 1
            if u < 0:
                break
            steps = self.items[u] * self.per_tile
            if steps == 0:
                continue
            for _ in range(steps):
                yield ("wait", self.s_full, t)
                yield ("wait", self.q_full[t % NSB], t // NSB)
                if t > 0:
                    yield ("wait", self.pt_free, t - 1)
                yield ("wait", self.dp_full, t)
                self.p_full.arrive()
                if t >= 1:
                    yield ("wait", self.dsm_free, t - 1)
                self.ds_full.arrive()
                if t > 0:
                    yield from drain(t - 1)
                t += 1
            yield ("wait", self.dkv_full, nit)
            nit += 1
        if t > 0:
            yield from drain(t - 1)

    def run(self):
        self.engine.run({"P": self.producer(), "S": self.s_issuer(), "D": self.dvdk_issuer(), "Q": self.dq_issuer(),
                         "C": self.compute()})


def _items(rng):
    n = rng.randrange(1, 14)
    return [rng.choice([0, 1, 1, 2, 3, 4, 5, 8, 8, 10]) for _ in range(n)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("drop", [False, True])
def test_backward_protocol_never_deadlocks_or_aliases(drop, d):
    rng = random.Random(20260 + drop + d)
    for trial in range(300):
        Sim(_items(rng), drop, random.Random(rng.random()), d=d).run()


@pytest.mark.parametrize("d", [64, 128])
def test_backward_protocol_single_and_empty_items(d):
    for items in ([1], [0], [0, 0, 1], [1, 0, 1, 0], [8], [1] * 12, [0] * 5 + [2]):
        for drop in (False, True):
            for seed in range(20):
                Sim(items, drop, random.Random(seed), d=d).run()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("plant", ["reduce_unstaged", "ring_too_deep"])
def test_planted_protocol_mistakes_are_caught(plant, d):
    rng = random.Random(7)
    caught = False
    for trial in range(200):
        try:
            Sim(_items(rng), False, random.Random(rng.random()), plant=plant, d=d).run()
        except ProtocolError:
            caught = True
            break
    assert caught
