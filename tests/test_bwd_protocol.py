"""Event simulation of the backward main kernel's barrier protocol (CPU).

The backward kernel runs four roles on one CTA's work: the TMA producer (K_j, V_j once per item,
Q_i / dO_i with their vectors into two stages), the MMA issuer, the elementwise warps (P^T, then
dS^T into TMEM and dS into shared memory) and the drain (reads each dQ tile out of TMEM; at the
end of an item stores dK, dV).  Products run on the tensor core in issue order, and a commit's
barrier completes once every product issued before it has finished.  The d = 128 issue order per
query tile g of an item: [S^T(g) for the item's first tile], dP^T(g), dV(g), [S^T(g + 1)], dK(g),
dQ^T(g).  TMEM holds S^T / P^T in one set of columns and dP^T / dS^T / dQ^T in another; dK and
dV accumulate in their own columns for a whole item.

The model is written from this description and from the waits and commits each role makes,
with random load and product latencies and random interleavings.  It checks:
- every wait finds its barrier with p or p + 1 completed phases (a parity wait for phase p
  is exact only then: with p - 1 it returns at once, with p + 2 never);
- every read of a TMEM region, a shared-memory stage or buffer finds the tile it expects
  (nothing is overwritten before its last reader is done, nothing is read before it is written);
- the dK / dV accumulators hold every query tile's contribution when the drain stores them;
- no deadlock.
A planted mistake in the waits (one phase off, or a wait left out) must fail a check.
"""
import random

import pytest


class Barrier:
    """Completion count and pending arrivals / bytes of one phase."""

    def __init__(self, name, count=1):
        self.name, self.count = name, count
        self.done = 0
        self.arrivals = 0
        self.tx = 0

    def arrive(self, tx=0):
        self.arrivals += 1
        self.tx += tx
        self._check()

    def complete_tx(self, tx):
        self.tx -= tx
        assert self.tx >= 0
        self._check()

    def _check(self):
        if self.arrivals == self.count and self.tx == 0:
            self.done += 1
            self.arrivals = 0

    def ready(self, phase):
        assert self.done in (phase, phase + 1), f"{self.name}: wait for phase {phase} found {self.done} completed"
        return self.done == phase + 1


class Sim:
    def __init__(self, items, rng, bug=None):
        self.items, self.rng, self.bug = items, rng, bug
        names = ["KFull", "KEmpty", "VFull", "VEmpty", "QFull0", "QFull1", "QEmpty0", "QEmpty1", "SFull", "DpFull",
                 "PReady", "DsReady", "DqFull", "DqFree", "DkvFull", "DkvEmpty"]
        self.bar = {n: Barrier(n) for n in names}
        # contents: name -> tag of the tile it holds
        self.mem = {"K": None, "V": None, "Q0": None, "Q1": None, "Scols": None, "DPcols": None, "dSsmem": None}
        self.accV = self.accK = None   # (item, query tiles accumulated) of dV and dK
        self.tc = []               # tensor core queue: ("mma", fn) or ("commit", barrier name)
        self.tma = []              # loads in flight: [delay, barrier, tx, region, tag]
        self.tiles = [(k, it) for k, n in enumerate(items) for it in range(n)]  # global tile g -> (item, index)

    def wait(self, name, phase):
        """Generator helper: block until barrier `name` completes phase `phase`."""
        while not self.bar[name].ready(phase):
            yield
        return

    def expect(self, region, tag):
        assert self.mem[region] == tag, f"{region} holds {self.mem[region]}, expected {tag}"

    # ------------------------------------------------------------------ asynchronous units
    def load(self, bar, region, tag):
        self.bar[bar].arrive(tx=1)
        self.mem[region] = ("loading", tag)          # a read before the copy lands fails
        self.tma.append([self.rng.randint(0, 8), bar, region, tag])

    def step_tma(self):
        for c in self.tma:
            c[0] -= 1
        for c in [c for c in self.tma if c[0] < 0]:
            self.tma.remove(c)
            _, bar, region, tag = c
            assert self.mem[region] == ("loading", tag), f"{region} changed under the copy of {tag}"
            self.mem[region] = tag
            self.bar[bar].complete_tx(1)

    def mma(self, reads, writes, update=None):
        """Queue a product: `reads` (region, tag) are checked when it starts and when it ends,
        `writes` (region, tag) hold a partial value in between."""
        self.tc.append(["mma", reads, writes, update, False])

    def commit(self, bar):
        self.tc.append(["commit", bar])

    def step_tensor_core(self):
        if not self.tc:
            return
        head = self.tc[0]
        if head[0] == "commit":
            self.bar[head[1]].arrive()
            self.tc.pop(0)
            return
        _, reads, writes, update, started = head
        for region, tag in reads:
            self.expect(region, tag)
        if not started:
            for region, tag in writes:
                self.mem[region] = ("writing", tag)
            head[4] = True
            return
        for region, tag in writes:
            self.mem[region] = tag
        if update:
            update()
        self.tc.pop(0)

    # ------------------------------------------------------------------ roles
    def loader(self):
        g = 0
        for k, n in enumerate(self.items):
            yield from self.wait("VEmpty", k - 1)
            self.load("VFull", "V", ("V", k))
            yield from self.load_q(g)
            yield from self.wait("KEmpty", k - 1)
            self.load("KFull", "K", ("K", k))
            for it in range(1, n):
                yield from self.load_q(g + it)
            g += n

    def load_q(self, g):
        st = g & 1
        yield from self.wait(f"QEmpty{st}", (g >> 1) - 1)
        self.load(f"QFull{st}", f"Q{st}", ("Q", g))    # Q_i, dO_i and the two vectors

    def issue_s(self, g, k):
        yield from self.wait(f"QFull{g & 1}", g >> 1)
        self.mma([("K", ("K", k)), (f"Q{g & 1}", ("Q", g))], [("Scols", ("S", g))])
        self.commit("SFull")

    def accumulate(self, which, k, it):
        def up():
            cur = getattr(self, which)
            assert cur == (None if it == 0 else (k, it)), f"{which} holds {cur} before query tile {it} of item {k}"
            setattr(self, which, (k, it + 1))
        return up

    def mma_issuer(self):
        bug = self.bug
        g = 0
        for k, n in enumerate(self.items):
            yield from self.wait("KFull", k)
            yield from self.wait("VFull", k)
            for it in range(n):
                st = g & 1
                q = (f"Q{st}", ("Q", g))
                if it == 0:
                    yield from self.issue_s(g, k)
                else:
                    yield from self.wait(f"QFull{st}", g >> 1)    # already waited when S^T(g) was issued
                # dP^T overwrites the columns the drain reads dQ^T(g - 1) from
                yield from self.wait("DqFree", g if bug == "dqfree_phase" else g - 1)
                self.mma([("V", ("V", k)), q], [("DPcols", ("dP", g))])
                self.commit("DpFull")
                if it == n - 1:
                    self.commit("VEmpty")
                yield from self.wait("PReady", g)
                if it == 0 and bug != "no_dkvempty_wait":
                    yield from self.wait("DkvEmpty", k - 1)
                self.mma([("Scols", ("P", g)), q], [], self.accumulate("accV", k, it))
                if bug == "qempty_early":
                    self.commit(f"QEmpty{st}")
                if it + 1 < n:
                    yield from self.issue_s(g + 1, k)
                yield from self.wait("DsReady", g)
                self.mma([("DPcols", ("dS", g)), q], [], self.accumulate("accK", k, it))
                if bug != "qempty_early":
                    self.commit(f"QEmpty{st}")
                self.mma([("dSsmem", ("dS", g)), ("K", ("K", k))], [("DPcols", ("dQ", g))])
                self.commit("DqFull")
                g += 1
            self.commit("KEmpty")
            self.commit("DkvFull")

    def elementwise(self):
        for g, (k, it) in enumerate(self.tiles):
            q = (f"Q{g & 1}", ("Q", g))                   # the stage's -L log2 e and -D vectors
            yield from self.wait("SFull", g)
            self.expect("Scols", ("S", g))
            self.expect(*q)
            self.mem["Scols"] = ("writing", ("P", g))
            if self.bug == "pready_early":
                self.bar["PReady"].arrive()
            yield
            self.mem["Scols"] = ("P", g)
            if self.bug != "pready_early":
                self.bar["PReady"].arrive()
            yield from self.wait("DpFull", g)
            # dQ(g - 1) has read the dS buffer.  The kernel waits for this, but DpFull(g) already
            # implies it: dQ(g - 1) is issued before dP^T(g), and a commit covers every earlier
            # product (the model passes without the wait as well).
            yield from self.wait("DqFull", g - 1)
            self.expect("DPcols", ("dP", g))
            self.expect(*q)
            self.mem["DPcols"] = ("writing", ("dS", g))
            self.mem["dSsmem"] = ("writing", ("dS", g))
            yield
            self.mem["DPcols"] = ("dS", g)
            self.mem["dSsmem"] = ("dS", g)
            self.bar["DsReady"].arrive()

    def drain(self):
        g = 0
        for k, n in enumerate(self.items):
            for it in range(n):
                yield from self.wait("DqFull", g)
                self.expect("DPcols", ("dQ", g))
                yield
                self.expect("DPcols", ("dQ", g))
                self.bar["DqFree"].arrive()
                g += 1
            yield from self.wait("DkvFull", k)
            assert self.accV == (k, n) and self.accK == (k, n), (k, n, self.accV, self.accK)
            yield
            assert self.accV == (k, n) and self.accK == (k, n), "dK / dV changed while the drain stored them"
            self.accV = self.accK = None
            self.bar["DkvEmpty"].arrive()

    def run(self):
        roles = [self.loader(), self.mma_issuer(), self.elementwise(), self.drain()]
        live = list(roles)
        for _ in range(200000):
            if not live and not self.tc and not self.tma:
                return
            r = self.rng.random()
            if r < 0.25:
                self.step_tma()
            elif r < 0.5:
                self.step_tensor_core()
            elif live:
                role = self.rng.choice(live)
                try:
                    next(role)
                except StopIteration:
                    live.remove(role)
        raise AssertionError("no progress (deadlock)")


def _random_items(rng):
    return [rng.randint(1, 6) for _ in range(rng.randint(1, 5))]


def test_protocol_random_work():
    rng = random.Random(2024)
    for _ in range(300):
        Sim(_random_items(rng), rng).run()


def test_single_tile_items():
    rng = random.Random(5)
    for n_items in range(1, 7):
        Sim([1] * n_items, rng).run()


@pytest.mark.parametrize("bug", ["dqfree_phase", "no_dkvempty_wait", "qempty_early", "pready_early"])
def test_planted_protocol_mistakes_are_caught(bug):
    """Each deliberate mistake in the model's waits or commits fails a check in some trial."""
    rng = random.Random(77)
    caught = 0
    for _ in range(300):
        try:
            Sim(_random_items(rng), rng, bug=bug).run()
        except AssertionError:
            caught += 1
    assert caught > 0, bug
