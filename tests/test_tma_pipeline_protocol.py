"""The barrier protocol of the TMA-fed NVFP4 GEMV (csrc/gemv_tma.cu), checked
on the CPU.

One producer thread per CTA streams ring stages (a full barrier per slot: its
arrive plus the stage's bytes); eight consumer warps wait for each stage,
decode it and arrive once each on the slot's empty barrier; the producer
refills a slot once all eight have released it.  The producer holds after
three stages until every consumer warp has staged the first group's x, keeps
its slot / phase count running across tiles and across the groups of a chain,
and the consumer warps meet at a barrier at each tile end and around each
group boundary.  mbarrier waits test only the parity of a phase, so a waiter
that could fall two phases behind would pass early.  This module replays the
schedule under random interleavings (bytes land in any order) and asserts
that every wait that passes has seen its target completion, every arrival
lands in its use's phase, and the run ends without a deadlock.  It also shows
that a schedule that lets the producer refill a slot released by only one
warp is caught.
"""
import random

import pytest

CW = 8
PREFETCH = 3


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.phase, self.pending, self.tx = name, count, 0, count, 0

    def arrive(self, use):
        assert self.phase == use, f"{self.name}: arrival for use {use} in phase {self.phase}"
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: too many arrivals"
        self.settle()

    def settle(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def passes(self, target):
        return (self.phase & 1) != (target & 1)


class Meet:
    """bar.sync among the consumer warps: use u opens when all CW have arrived."""

    def __init__(self):
        self.arrived = {}

    def arrive(self, use):
        self.arrived[use] = self.arrived.get(use, 0) + 1

    def open(self, use):
        return self.arrived.get(use, 0) >= CW


def simulate(S, tiles, nst, groups, seed, empty_count=CW):
    rnd = random.Random(seed)
    full = [Bar(f"full[{s}]", 1) for s in range(S)]
    empty = [Bar(f"empty[{s}]", empty_count) for s in range(S)]
    meet = Meet()
    staged = [0]
    total = groups * tiles * nst

    prod = []
    for i in range(total):
        s, u = i % S, i // S
        if i >= S:
            prod.append(("wait", empty[s], u - 1))
        prod.append(("tma", full[s], u))
        if i + 1 == PREFETCH:
            prod.append(("hold", None, None))
    progs = {"producer": prod}
    for w in range(CW):
        ops, i, m = [], 0, 0
        for p in range(groups):
            if p > 0:                                    # y of the earlier groups before x is read
                ops += [("meet_arrive", None, m), ("meet_wait", None, m)]
                m += 1
                ops += [("meet_arrive", None, m), ("meet_wait", None, m)]
                m += 1
            if p == 0:
                ops.append(("staged", None, None))
            for _ in range(tiles):
                for _ in range(nst):
                    s, u = i % S, i // S
                    ops += [("wait", full[s], u), ("arrive", empty[s], u)]
                    i += 1
                ops += [("meet_arrive", None, m), ("meet_wait", None, m)]   # tile end
                m += 1
        progs[f"warp{w}"] = ops

    pc = {k: 0 for k in progs}
    landing = []

    def ready(op):
        kind, bar, n = op
        if kind == "wait":
            return bar.passes(n)
        if kind == "hold":
            return staged[0] >= CW
        if kind == "meet_wait":
            return meet.open(n)
        return True

    for _ in range(1000000):
        cand = [k for k, ops in progs.items() if pc[k] < len(ops) and ready(ops[pc[k]])]
        if landing:
            cand.append("landing")
        if not cand:
            assert all(pc[k] == len(ops) for k, ops in progs.items()), "deadlock"
            return
        k = rnd.choice(cand)
        if k == "landing":
            bar = landing.pop(rnd.randrange(len(landing)))
            bar.tx -= 1
            bar.settle()
            continue
        kind, bar, n = progs[k][pc[k]]
        pc[k] += 1
        if kind == "wait":
            assert bar.phase >= n + 1, f"{k}: wait for {bar.name} #{n} passed in phase {bar.phase}"
        elif kind == "arrive":
            bar.arrive(n)
        elif kind == "tma":
            assert bar.phase == n, f"{bar.name}: expect_tx for use {n} in phase {bar.phase}"
            bar.tx += 1
            bar.arrive(n)
            landing.append(bar)
        elif kind == "staged":
            staged[0] += 1
        elif kind == "meet_arrive":
            meet.arrive(n)
    raise AssertionError("no progress")


@pytest.mark.parametrize("S", [3, 4, 5, 8])
def test_tma_schedule_never_skips_a_phase(S):
    for tiles in (1, 2, 3):
        for nst in (1, 2, 7):
            for groups in (1, 2, 3):
                for seed in range(6):
                    simulate(S, tiles, nst, groups, seed)


def test_single_release_schedule_is_caught():
    """If a slot counted as empty after ONE warp released it, the producer
    could refill it while other warps still wait for the older use."""
    with pytest.raises(AssertionError, match="passed in phase|arrival for use"):
        for seed in range(300):
            simulate(3, 3, 2, 1, seed, empty_count=1)
