"""The grid-wide barrier of the GEMV chain (csrc/gemv_tma.cu, grid_barrier),
model-checked on the CPU.

One thread per CTA runs: read the generation word, add one to the count; the
CTA whose add returns grid - 1 resets the count and then bumps the
generation, the others spin until the generation differs from what they read.
The two words live in caller memory and are reused by every barrier of every
launch and graph replay.  Each atomic step is one scheduling point here, in
random order, across several consecutive barriers and several launches that
reuse the words.  Asserted: no CTA leaves barrier b before every CTA has
arrived at it; the words end each launch at count 0 with the generation
advanced by the number of barriers; no run deadlocks.  A variant that reads
the generation after its add (the wrong order) is caught.
"""
import random

import pytest


def run_launch(words, ctas, barriers, rnd, read_after_add=False):
    """One launch: every CTA passes `barriers` barriers in turn."""
    gen0 = words["gen"]
    arrived = [0] * barriers          # CTAs that have added to the count at barrier b
    state = [("start", 0, None) for _ in range(ctas)]    # (step, barrier, my_gen)
    done = [False] * ctas
    for _ in range(100000):
        live = [c for c in range(ctas) if not done[c]]
        if not live:
            assert words["count"] == 0
            assert words["gen"] == gen0 + barriers
            return
        movable = []
        for c in live:
            step, b, my = state[c]
            if step == "spin" and words["gen"] == my:
                continue
            movable.append(c)
        assert movable, "deadlock"
        c = rnd.choice(movable)
        step, b, my = state[c]
        if step == "start":
            if read_after_add:
                state[c] = ("add", b, None)
            else:
                state[c] = ("add", b, words["gen"])          # ld.acquire of the generation
        elif step == "add":
            old = words["count"]
            words["count"] += 1                               # atomicAdd
            arrived[b] += 1
            if old == ctas - 1:
                state[c] = ("reset", b, my)
            elif read_after_add:
                state[c] = ("read", b, None)                  # the generation read, a step of its own
            else:
                state[c] = ("spin", b, my)
        elif step == "read":
            state[c] = ("spin", b, words["gen"])
        elif step == "reset":
            words["count"] = 0                                # atomicExch
            state[c] = ("bump", b, my)
        elif step == "bump":
            words["gen"] += 1                                 # atomicAdd, after the fence
            state[c] = ("leave", b, my)
        elif step in ("spin", "leave"):
            assert arrived[b] == ctas, f"CTA {c} left barrier {b} with {arrived[b]} of {ctas} arrived"
            if b + 1 == barriers:
                done[c] = True
            else:
                state[c] = ("start", b + 1, None)
    raise AssertionError("no progress")


@pytest.mark.parametrize("ctas", [1, 2, 3, 5, 8])
def test_grid_barrier_is_safe_and_reusable(ctas):
    for seed in range(60):
        rnd = random.Random(seed)
        words = {"count": 0, "gen": 0}
        for launch in range(3):                               # the words carry over between launches
            run_launch(words, ctas, barriers=1 + (seed + launch) % 3, rnd=rnd)


def test_reading_the_generation_after_the_add_is_caught():
    """Reading the generation after the add lets a CTA see the bump of the
    barrier it is in (or of the next one) as its own baseline: it then spins
    forever or leaves early; the model reports either."""
    with pytest.raises(AssertionError, match="deadlock|left barrier"):
        for seed in range(400):
            rnd = random.Random(seed)
            words = {"count": 0, "gen": 0}
            run_launch(words, 4, barriers=3, rnd=rnd, read_after_add=True)


def run_launch_with_abort(words, ctas, aborting, rnd):
    """One launch with one barrier in which CTA `aborting` gives up before it
    arrives (its own bounded wait ran out, or the abort flag was raised).
    The others add, spin, and leave when their spin limit runs out: in the
    model, when nothing else can move.  Returns the CTAs that left through
    the timeout."""
    state = {c: "start" for c in range(ctas) if c != aborting}
    my_gen = {}
    timed_out = set()
    while state:
        movable = [c for c, st in state.items() if not (st == "spin" and words["gen"] == my_gen[c])]
        if not movable:                                       # every spinner's limit runs out
            timed_out.update(state)
            return timed_out
        c = rnd.choice(movable)
        st = state[c]
        if st == "start":
            my_gen[c] = words["gen"]
            state[c] = "add"
        elif st == "add":
            old = words["count"]
            words["count"] += 1
            state[c] = "reset" if old == ctas - 1 else "spin"
        elif st == "reset":
            words["count"] = 0
            state[c] = "bump"
        elif st == "bump":
            words["gen"] += 1
            del state[c]
        else:
            del state[c]
    return timed_out


@pytest.mark.parametrize("ctas", [2, 3, 5])
def test_an_aborted_barrier_leaves_the_words_dirty_until_the_caller_zeroes_them(ctas):
    """After a Q4_ETIMEOUT the count holds the CTAs that did arrive, so a next
    launch on the same words can release a barrier early, hang, or leave the
    count non-zero again: the header therefore requires the caller to zero
    both words after any Q4_ETIMEOUT.  Once zeroed, the words work again."""
    wrong = 0
    for seed in range(40):
        rnd = random.Random(seed)
        words = {"count": 0, "gen": 0}
        run_launch(words, ctas, barriers=2, rnd=rnd)
        timed_out = run_launch_with_abort(words, ctas, aborting=seed % ctas, rnd=rnd)
        assert len(timed_out) == ctas - 1 and words["count"] == ctas - 1
        try:
            run_launch(dict(words), ctas, barriers=1, rnd=random.Random(seed))
        except AssertionError:
            wrong += 1
        words = {"count": 0, "gen": 0}                        # the caller's re-zeroing
        run_launch(words, ctas, barriers=2, rnd=rnd)
    assert wrong > 0
