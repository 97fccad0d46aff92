"""Model check (CPU) of the stream kernel's shared-memory ring protocol.

The stream kernel's producer lane and its consumer groups synchronise through
full/empty mbarriers waited on by phase parity.  This test replays the
protocol in a small Python model under many random interleavings of the
producer, the consumer groups and the completion of bulk copies, with the
mbarrier rules as PTX defines them: a barrier's phase completes once its
expected arrivals (and, for "full", the armed transaction bytes) are in;
try_wait.parity(P) succeeds when the current phase's parity differs from P.

It checks that every wait passes only when the awaited fill has really landed
(and holds the row and slice the consumer expects), that the producer never
re-arms a barrier whose phase is still open, and that every schedule finishes.
The same model run with one ring shared by all groups -- groups stepping over
each other's slots -- must be caught, since a group can then reach a slot one
fill ahead of another group and see the earlier phase's parity.
"""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count = count
        self.phase = 0
        self.arrived = 0
        self.tx = 0

    def try_wait(self, parity):
        return (self.phase & 1) != parity

    def arrive(self, tx=0):
        self.arrived += 1
        self.tx += tx
        self._maybe_complete()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._maybe_complete()

    def _maybe_complete(self):
        assert self.arrived <= self.count, "more arrivals than expected in one phase"
        if self.arrived == self.count and self.tx == 0:
            self.phase += 1
            self.arrived = 0


def simulate(rows, nslices, slots, groups, shared_ring, rng):
    S = slots
    full = [Barrier(1) for _ in range(S)]
    empty = [Barrier(1) for _ in range(S)]          # one arrival stands for the group's warps
    content = [None] * S
    inflight = []                                   # (slot, (row, k))
    SG = S // groups

    # producer state
    prod = {"i": 0, "k": 0, "used": [0] * groups, "n": 0}

    def prod_slot():
        i, k = prod["i"], prod["k"]
        if shared_ring:
            n = prod["n"]
            return n % S, (n // S) & 1
        g = i % groups
        n = prod["used"][g]
        return g * SG + n % SG, (n // SG) & 1

    # consumer state per group: next own row index, slice, ring position
    cons = []
    for g in range(groups):
        cons.append({"i": g, "k": 0, "lslot": 0, "ph": 0, "gslot": 0, "gph": 0, "done": g >= rows})
        if shared_ring:
            # step over the rows of other groups before the first own row
            n = g * nslices
            cons[g]["gslot"], cons[g]["gph"] = n % S, (n // S) & 1

    def cons_slot(c, g):
        if shared_ring:
            return c["gslot"], c["gph"]
        return g * SG + c["lslot"], c["ph"]

    steps = 0
    while True:
        steps += 1
        assert steps < 100000, "no progress (deadlock)"
        actions = []
        if prod["i"] < rows:
            slot, ph = prod_slot()
            if empty[slot].try_wait(ph ^ 1):
                actions.append("prod")
        for g, c in enumerate(cons):
            if not c["done"]:
                slot, ph = cons_slot(c, g)
                if full[slot].try_wait(ph):
                    actions.append(("cons", g))
        if inflight:
            actions.append("copy")
        if not actions:
            if prod["i"] >= rows and all(c["done"] for c in cons) and not inflight:
                return
            raise AssertionError("deadlock")
        a = rng.choice(actions)
        if a == "prod":
            slot, ph = prod_slot()
            assert full[slot].arrived == 0 and full[slot].tx == 0, "re-armed an open phase"
            full[slot].arrive(tx=16)
            inflight.append((slot, (prod["i"], prod["k"])))
            if shared_ring:
                prod["n"] += 1
            else:
                prod["used"][prod["i"] % groups] += 1
            prod["k"] += 1
            if prod["k"] == nslices:
                prod["k"] = 0
                prod["i"] += 1
        elif a == "copy":
            slot, what = inflight.pop(rng.randrange(len(inflight)))
            content[slot] = what
            full[slot].complete_tx(16)
        else:
            g = a[1]
            c = cons[g]
            slot, ph = cons_slot(c, g)
            assert content[slot] == (c["i"], c["k"]), f"group {g} read {content[slot]}, wanted {(c['i'], c['k'])}"
            content[slot] = None
            empty[slot].arrive()
            if shared_ring:
                n = c["gslot"] + 1
                c["gslot"], c["gph"] = (0, c["gph"] ^ 1) if n == S else (n, c["gph"])
            else:
                c["lslot"] += 1
                if c["lslot"] == SG:
                    c["lslot"], c["ph"] = 0, c["ph"] ^ 1
            c["k"] += 1
            if c["k"] == nslices:
                c["k"] = 0
                c["i"] += groups
                if shared_ring:
                    # step over the other groups' rows
                    for _ in range((groups - 1) * nslices):
                        n = c["gslot"] + 1
                        c["gslot"], c["gph"] = (0, c["gph"] ^ 1) if n == S else (n, c["gph"])
                if c["i"] >= rows:
                    c["done"] = True


CASES = [  # (rows, nslices, slots, groups): shapes of H = 7168 / 4096 / 1024 / 16384 workloads
    (31, 9, 16, 2), (31, 3, 16, 2), (27, 5, 28, 3), (12, 9, 32, 4), (9, 17, 7, 1), (5, 3, 28, 3), (40, 2, 32, 4),
]


@pytest.mark.parametrize("rows,nslices,slots,groups", CASES)
def test_per_group_sub_rings_are_safe(rows, nslices, slots, groups):
    rng = random.Random(1234)
    for _ in range(150):
        simulate(rows, nslices, slots, groups, shared_ring=False, rng=rng)


def test_one_shared_ring_is_caught():
    rng = random.Random(99)
    caught = 0
    for _ in range(1500):
        try:
            simulate(31, 9, 16, 2, shared_ring=True, rng=rng)
        except AssertionError:
            caught += 1
    assert caught > 0
