"""The barrier protocol of the tensor-core small-batch GEMM, checked on the CPU.

The kernel's roles (eight decode warps in two warpgroups, each warp arriving
once per stage and per slot, the MMA thread, the weight-slot TMA thread and
the X-tile TMA thread) hand stages to each other through
mbarriers whose waits test only the parity of a phase.  A waiter that can
fall two phases behind a barrier is fooled: the wait for completion #u
passes as soon as completion #u-2 has happened.  This module replays the
kernel's schedule (the same ring sizes and stage/slot arithmetic as the
kernel's Cfg) under random interleavings, with asynchronous MMA completion
and TMA landing, and asserts that

  * every wait that passes has really seen its target completion, and
  * every arrival lands in the phase of the use it belongs to.

It also shows that the schedule in which the two warpgroups take alternate
weight slots over one shared stage ring is caught by the same check (the
case that faulted on the GPU at batch 128).
"""
import random

import pytest

TMEM_COLS, A_COLS = 256, 32
DEC_WARPS = 8


def rings(MB):
    """(stages, weight slots) of the kernel for batch tile MB."""
    dcols = max(32, MB)
    ns = (TMEM_COLS - dcols) // A_COLS
    nw = 3 if MB == 64 else 2
    return ns, nw


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
        """The hardware test: the phase with the target's parity is not current."""
        return (self.phase & 1) != (target & 1)


def simulate(MB, nslots, seed, alternate_slots=False):
    rnd = random.Random(seed)
    ns, nw = rings(MB)
    nst = 4 * nslots
    warps_per_stage = DEC_WARPS // 2 if alternate_slots else DEC_WARPS
    a_full = [Bar(f"a_full[{s}]", warps_per_stage + 1) for s in range(ns)]
    a_empty = [Bar(f"a_empty[{s}]", 1) for s in range(ns)]
    w_full = [Bar(f"w_full[{s}]", 1) for s in range(nw)]
    w_empty = [Bar(f"w_empty[{s}]", warps_per_stage) for s in range(nw)]
    done = Bar("done", 1)

    progs = {}
    for wp in range(DEC_WARPS):
        g = wp // 4                    # the warp's warpgroup
        ops = []
        slots = range(g, nslots, 2) if alternate_slots else range(nslots)
        for j in slots:
            ops.append(("wait", w_full[j % nw], j // nw))
            for c in range(4):
                i = 4 * j + c
                if c == 3:
                    ops.append(("arrive", w_empty[j % nw], j // nw))
                if i >= ns:
                    ops.append(("wait", a_empty[i % ns], i // ns - 1))
                ops.append(("arrive", a_full[i % ns], i // ns))
        progs[f"decode{wp}"] = ops
    ops = []
    for i in range(nst):
        ops += [("wait", a_full[i % ns], i // ns), ("mma", a_empty[i % ns], i // ns)]
    progs["mma"] = ops + [("mma", done, 0)]
    ops = []
    for j in range(nslots):
        if j >= nw:
            ops.append(("wait", w_empty[j % nw], j // nw - 1))
        ops.append(("tma", w_full[j % nw], j // nw))
    progs["weights"] = ops
    ops = []
    for i in range(nst):
        if i >= ns:
            ops.append(("wait", a_empty[i % ns], i // ns - 1))
        ops.append(("tma", a_full[i % ns], i // ns))
    progs["x"] = ops

    pc = {k: 0 for k in progs}
    tensor, landing = [], []       # MMAs complete in order; copies land in any order
    for _ in range(400000):
        ready = []
        for k, ops in progs.items():
            if pc[k] < len(ops):
                op = ops[pc[k]]
                if op[0] != "wait" or op[1].passes(op[2]):
                    ready.append(k)
        if tensor:
            ready.append("tensor")
        if landing:
            ready.append("landing")
        if not ready:
            assert all(pc[k] == len(ops) for k, ops in progs.items()), "deadlock"
            assert done.phase == 1
            return
        k = rnd.choice(ready)
        if k == "tensor":
            bar, use = tensor.pop(0)
            bar.arrive(use)
            continue
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
        elif kind == "mma":
            tensor.append((bar, n))
        else:                      # arrive.expect_tx, then the bytes land later
            assert bar.phase == n, f"{bar.name}: expect_tx for use {n} in phase {bar.phase}"
            bar.tx += 1
            bar.arrive(n)
            landing.append(bar)
    raise AssertionError("no progress")


@pytest.mark.parametrize("MB", [16, 32, 64, 128])
def test_kernel_schedule_never_skips_a_phase(MB):
    for nslots in range(1, 9):
        for seed in range(25):
            simulate(MB, nslots, seed)


def test_alternate_slot_schedule_is_caught():
    """Alternating warpgroups over a 4-stage ring (batch 128) let one group
    reach a stage two uses ahead of the barrier: the check must fire."""
    with pytest.raises(AssertionError, match="passed in phase"):
        for seed in range(400):
            simulate(128, 4, seed, alternate_slots=True)
