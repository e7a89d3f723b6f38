"""Event simulation of the forward kernel's K/V ring protocol with paired barriers (CPU).

The forward's loader streams key/value tiles through a ring of S shared-memory slots in the
token order K_0 (first item), then per step V_j, K_{j+1}, and across an item boundary
V_{n-1}, K_0 of the next item.  With the static work list it lands each V and the K after it on
one "full" barrier (the V slot's), which expects both tiles; the MMA warp waits once per step
and releases each pair with one commit on the V slot's "empty" barrier.  The pair spanning an
item boundary is released after the next item's first S products, and the CTA's last V expects
a single tile.  The loader waits, before refilling a slot, on the pair released there before
(and on the release of the lone first K for the slot it occupied).

Barrier waits in the kernel test a phase by its parity.  That is exact only while the barrier
is at most one phase ahead of the waiter: a wait for phase p must find the barrier with p or
p + 1 completed phases.  With p - 1 it would return at once (the previous phase has the other
parity), and with p + 2 it would never return.  The simulation runs the loader and the MMA
warp as two processes, with random load latencies and random interleavings, and checks:
- every wait finds its barrier with p or p + 1 completed phases;
- a tile is never overwritten before the MMA warp has released it;
- the MMA warp never reads a slot whose tile has not landed, or that holds another token;
- the protocol never deadlocks.
The model is written from the protocol's description, not from the kernel's code.
"""
import random

import pytest


class Barrier:
    """Completion count, pending arrivals and pending bytes of one phase."""

    def __init__(self, count):
        self.count = count
        self.done = 0          # completed phases
        self.arrivals = 0
        self.tx = 0

    def arrive_expect(self, tx):
        self.arrivals += 1
        self.tx += tx
        self._check()

    def complete_tx(self, tx):
        self.tx -= tx
        assert self.tx >= 0
        self._check()

    def arrive(self):
        self.arrivals += 1
        self._check()

    def _check(self):
        if self.arrivals == self.count and self.tx == 0:
            self.done += 1
            self.arrivals = 0

    def ready(self, phase):
        """The kernel's parity wait for `phase`, with the aliasing check."""
        assert self.done in (phase, phase + 1), f"wait for phase {phase} found {self.done} completed"
        return self.done == phase + 1


def tokens_of(items):
    """Token list: (kind, item index, step) in the loader's order."""
    out = []
    for i, n in enumerate(items):
        for j in range(n):
            out.append(("K", i, j))
            out.append(("V", i, j))
    return out


def simulate(items, S, rng, bug=None):
    toks = tokens_of(items)
    T = len(toks)
    full = [Barrier(1) for _ in range(S)]
    empty = [Barrier(1) for _ in range(S)]
    slot_tok = [None] * S          # token index whose tile the slot holds (or is receiving)
    landed = [False] * S
    released = set()               # tokens the MMA warp has released
    in_flight = []                 # (remaining delay, token)

    # loader state
    lt = 0
    # MMA state: which item / step, and what it waits for next
    m_item, m_step, m_phase = 0, -1, "start"
    m_tok = 0
    pending = None                 # V token whose pair (with the next item's K_0) is not yet released

    def first_of_pair(t):
        return t > 0 and t % 2 == 1

    def full_bar(t):
        return t % S if (t == 0 or first_of_pair(t)) else (t - 1) % S

    def pair_phase(t):
        return t // S

    def release(vt):
        # one commit frees the V slot and the slot of the token after it
        empty[vt % S].arrive()
        released.add(vt)
        if vt + 1 < T:
            released.add(vt + 1)

    steps = 0
    while True:
        steps += 1
        assert steps < 200000, "no progress"
        # 1. land copies in flight
        nxt = []
        for d, t in in_flight:
            if d <= 0:
                s = t % S
                assert slot_tok[s] == t
                landed[s] = True
                full[full_bar(t)].complete_tx(1)
            else:
                nxt.append((d - 1, t))
        in_flight = nxt
        # 2. loader: next token, if its slot is free
        if lt < T and rng.random() < 0.7:
            s = lt % S
            need_wait = lt >= S and (first_of_pair(lt) or (lt == S and bug != "skip_lone_k_wait"))
            ok = True
            if need_wait:
                ok = empty[s].ready(pair_phase(lt) - 1)
            if ok:
                prev = lt - S
                if prev >= 0:
                    assert prev in released, f"token {lt} would overwrite unreleased token {prev}"
                slot_tok[s] = lt
                landed[s] = False
                if lt == 0:
                    full[0].arrive_expect(1)
                elif first_of_pair(lt):
                    # a V expects its K partner too, except the CTA's last V
                    full[s].arrive_expect(2 if lt + 1 < T and bug != "single_expect" else 1)
                in_flight.append((rng.randint(0, 6), lt))
                lt += 1
        # 3. MMA warp
        if m_item < len(items) and rng.random() < 0.7:
            n = items[m_item]
            if m_phase == "start":
                # item start: K_0 (waited only for the very first token)
                k0 = m_tok
                if k0 == 0:
                    if not full[0].ready(0):
                        continue
                assert slot_tok[k0 % S] == k0 and landed[k0 % S], "K_0 read before it landed"
                m_tok += 1
                if pending is not None:
                    release(pending)    # the boundary pair: its K_0 has now been read
                    pending = None
                else:
                    empty[k0 % S].arrive()
                    released.add(k0)
                m_phase, m_step = "step", 0
            else:
                vt = m_tok
                if not full[vt % S].ready(pair_phase(vt)):
                    continue
                assert slot_tok[vt % S] == vt and landed[vt % S], "V read before it landed"
                has_k = m_step + 1 < n
                if has_k:
                    kt = vt + 1
                    assert slot_tok[kt % S] == kt and landed[kt % S], "K read before it landed"
                    m_tok += 2
                    release(vt)
                else:
                    m_tok += 1
                    if bug == "release_boundary_early":
                        release(vt)
                    else:
                        pending = vt
                m_step += 1
                if m_step == n:
                    m_item += 1
                    m_phase = "start"
        if m_item == len(items) and lt == T and not in_flight:
            break
    if pending is not None:
        release(pending)
    assert m_tok == T


@pytest.mark.parametrize("S", [4, 6])
def test_paired_ring_random_work(S):
    rng = random.Random(1234 + S)
    for trial in range(300):
        n_items = rng.randint(1, 6)
        items = [rng.randint(1, 9) for _ in range(n_items)]
        simulate(items, S, rng)


def test_single_tile_items():
    rng = random.Random(7)
    for S in (4, 6):
        for n_items in range(1, 8):
            simulate([1] * n_items, S, rng)


@pytest.mark.parametrize("bug", ["skip_lone_k_wait", "release_boundary_early", "single_expect"])
def test_planted_protocol_mistakes_are_caught(bug):
    """Each deliberate protocol mistake in the model fails one of the checks in some trial."""
    rng = random.Random(99)
    caught = 0
    for trial in range(300):
        items = [rng.randint(1, 9) for _ in range(rng.randint(1, 6))]
        try:
            simulate(items, 4, rng, bug=bug)
        except AssertionError:
            caught += 1
    assert caught > 0, bug


def test_parity_alias_is_detected():
    """The check itself: a wait two phases ahead of its barrier must fail."""
    b = Barrier(1)
    b.arrive()
    with pytest.raises(AssertionError):
        b.ready(2)
